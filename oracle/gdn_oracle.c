/*
 * fp64 CPU oracle for draft-tree verification of a Gated DeltaNet layer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library path links, loads or calls this
 * file; only the tests, the smoke check and the CPU-baseline leg of the benchmark do.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes is the plain definition, with no WY transform, blocking or reordering:
 *
 *   gated delta rule  S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,  o_t = S_t q_t
 *   (S is d_v x d_k; a_t = exp(g_t)).
 *
 * For a draft tree (GDN Tree-Scan abstract: every candidate row must carry the recurrent
 * state that native sequential decode would produce along its root-to-node path) each node's
 * output is obtained by replaying the rule from the committed state S_0 along the node's
 * root-to-node path. A branch therefore never sees another branch (TreeWY page, method
 * section: each candidate refers only to its common ancestors).
 *
 * The pseudo-value of node t (TreeWY page, method section: the new value minus what the
 * preceding state already predicts) is read off the last replay step:
 *   u_t = b_t (v_t - a_t S_{parent(t)} k_t),  so that  S_t = a_t S_{parent(t)} + u_t k_t^T.
 * G_t is the cumulative log-gate sum over the root-to-node path.
 *
 * Commit (TreeWY page, method section: only the accepted path's state is rebuilt) is the
 * same replay along the accepted path; an empty path keeps S_0.
 *
 * Layouts match the library's: ST0 [B][H][d_k][d_v] (= S transposed), q,k [T][H][d_k],
 * v [T][H][d_v], beta,g [T][H], parent [T] request-local (-1 = child of the committed
 * state), cu_nodes [B+1], path [B][max_path], path_len [B]. All floating inputs are fp64.
 *
 * Outputs are compact over the listed (request, head) pairs: pair i (in list order)
 * contributes n_nodes(r) rows to o_c/U_c/G_c, and one d_k x d_v block to ST_c.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_TREE 1
#define ORACLE_BAD_PATH 2
#define ORACLE_BAD_ARG 3

/* Tree check: parent[t] in [-1, t-1] for every node of every request. */
static int check_tree(int B, const int *parent, const int *cu_nodes) {
    for (int r = 0; r < B; ++r) {
        int t0 = cu_nodes[r], n = cu_nodes[r + 1] - cu_nodes[r];
        if (n < 0) return ORACLE_BAD_ARG;
        for (int t = 0; t < n; ++t) {
            int p = parent[t0 + t];
            if (p < -1 || p >= t) return ORACLE_BAD_TREE;
        }
    }
    return ORACLE_OK;
}

/* Accepted path check: root first, each next node a child of the previous one. */
static int check_path(int B, const int *parent, const int *cu_nodes, const int *path,
                      const int *path_len, int max_path) {
    for (int r = 0; r < B; ++r) {
        int t0 = cu_nodes[r], n = cu_nodes[r + 1] - cu_nodes[r];
        int L = path_len[r];
        if (L < 0 || L > max_path || L > n) return ORACLE_BAD_PATH;
        int prev = -1;
        for (int i = 0; i < L; ++i) {
            int x = path[(size_t)r * max_path + i];
            if (x < 0 || x >= n) return ORACLE_BAD_PATH;
            if (parent[t0 + x] != prev) return ORACLE_BAD_PATH;
            prev = x;
        }
    }
    return ORACLE_OK;
}

/* One step of the rule on S (d_v x d_k, row-major S[i*dk + j]) for node (t, h).
 * Writes the pseudo-value u (length d_v) before S is overwritten. */
static void rule_step(double *S, int dk, int dv, double a, double b, const double *kv,
                      const double *vv, double *Sk, double *u) {
    /* Sk = S k */
    for (int i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * kv[j];
        Sk[i] = acc;
    }
    /* S <- a S (I - b k k^T) + b v k^T = a S - a b (S k) k^T + b v k^T */
    for (int i = 0; i < dv; ++i) {
        u[i] = b * (vv[i] - a * Sk[i]);
        double c = -a * b * Sk[i] + b * vv[i];
        for (int j = 0; j < dk; ++j) S[(size_t)i * dk + j] = a * S[(size_t)i * dk + j] + c * kv[j];
    }
}

static void load_S0(double *S, const double *ST0, int r, int h, int H, int dk, int dv) {
    const double *src = ST0 + ((size_t)r * H + h) * (size_t)dk * dv;
    for (int j = 0; j < dk; ++j)
        for (int i = 0; i < dv; ++i) S[(size_t)i * dk + j] = src[(size_t)j * dv + i];
}

static int pair_at(const int *pair_list, int idx) { return pair_list ? pair_list[idx] : idx; }

int gdn_oracle_verify(int B, int H, int dk, int dv, const double *ST0, const double *q,
                      const double *k, const double *v, const double *beta, const double *g,
                      const int *parent, const int *cu_nodes, const int *pair_list, int n_pairs,
                      double *o_c, double *U_c, double *G_c, int n_threads) {
    if (B < 0 || H <= 0 || dk <= 0 || dv <= 0) return ORACLE_BAD_ARG;
    int rc = check_tree(B, parent, cu_nodes);
    if (rc) return rc;
    if (!pair_list) n_pairs = B * H;
    /* compact row offsets per listed pair */
    size_t *row0 = (size_t *)malloc(sizeof(size_t) * (size_t)(n_pairs + 1));
    if (!row0) return ORACLE_BAD_ARG;
    row0[0] = 0;
    int max_n = 1;
    for (int r = 0; r < B; ++r)
        if (cu_nodes[r + 1] - cu_nodes[r] > max_n) max_n = cu_nodes[r + 1] - cu_nodes[r];
    for (int i = 0; i < n_pairs; ++i) {
        int p = pair_at(pair_list, i);
        if (p < 0 || p >= B * H) { free(row0); return ORACLE_BAD_ARG; }
        int r = p / H;
        row0[i + 1] = row0[i] + (size_t)(cu_nodes[r + 1] - cu_nodes[r]);
    }
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#endif
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
        double *Sk = (double *)malloc(sizeof(double) * (size_t)dv);
        double *u = (double *)malloc(sizeof(double) * (size_t)dv);
        int *stack = (int *)malloc(sizeof(int) * (size_t)max_n);
#pragma omp for schedule(dynamic, 1)
        for (int i = 0; i < n_pairs; ++i) {
            int p = pair_at(pair_list, i);
            int r = p / H, h = p % H;
            int t0 = cu_nodes[r], n = cu_nodes[r + 1] - cu_nodes[r];
            for (int t = 0; t < n; ++t) {
                /* root-to-node path: walk parents, then replay from the root */
                int m = 0;
                for (int x = t; x >= 0; x = parent[t0 + x]) stack[m++] = x;
                load_S0(S, ST0, r, h, H, dk, dv);
                double Gsum = 0.0;
                for (int s = m - 1; s >= 0; --s) {
                    size_t th = (size_t)(t0 + stack[s]) * H + h;
                    double gj = g[th];
                    double a = exp(gj);
                    Gsum += gj;
                    rule_step(S, dk, dv, a, beta[th], k + th * dk, v + th * dv, Sk, u);
                }
                size_t th = (size_t)(t0 + t) * H + h;
                const double *qv = q + th * dk;
                size_t row = row0[i] + (size_t)t;
                for (int a = 0; a < dv; ++a) {
                    double acc = 0.0;
                    for (int j = 0; j < dk; ++j) acc += S[(size_t)a * dk + j] * qv[j];
                    o_c[row * dv + a] = acc;
                    U_c[row * dv + a] = u[a];
                }
                G_c[row] = Gsum;
            }
        }
        free(S); free(Sk); free(u); free(stack);
    }
    free(row0);
    return ORACLE_OK;
}

int gdn_oracle_commit(int B, int H, int dk, int dv, const double *ST0, const double *k,
                      const double *v, const double *beta, const double *g, const int *parent,
                      const int *cu_nodes, const int *path, const int *path_len, int max_path,
                      const int *pair_list, int n_pairs, double *ST_c, int n_threads) {
    if (B < 0 || H <= 0 || dk <= 0 || dv <= 0 || max_path < 0) return ORACLE_BAD_ARG;
    int rc = check_tree(B, parent, cu_nodes);
    if (rc) return rc;
    rc = check_path(B, parent, cu_nodes, path, path_len, max_path);
    if (rc) return rc;
    if (!pair_list) n_pairs = B * H;
    for (int i = 0; i < n_pairs; ++i) {
        int p = pair_at(pair_list, i);
        if (p < 0 || p >= B * H) return ORACLE_BAD_ARG;
    }
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#endif
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
        double *Sk = (double *)malloc(sizeof(double) * (size_t)dv);
        double *u = (double *)malloc(sizeof(double) * (size_t)dv);
#pragma omp for schedule(dynamic, 1)
        for (int i = 0; i < n_pairs; ++i) {
            int p = pair_at(pair_list, i);
            int r = p / H, h = p % H;
            int t0 = cu_nodes[r];
            load_S0(S, ST0, r, h, H, dk, dv);
            for (int s = 0; s < path_len[r]; ++s) {
                size_t th = (size_t)(t0 + path[(size_t)r * max_path + s]) * H + h;
                rule_step(S, dk, dv, exp(g[th]), beta[th], k + th * dk, v + th * dv, Sk, u);
            }
            double *dst = ST_c + (size_t)i * dk * dv;
            for (int j = 0; j < dk; ++j)
                for (int a = 0; a < dv; ++a) dst[(size_t)j * dv + a] = S[(size_t)a * dk + j];
        }
        free(S); free(Sk); free(u);
    }
    return ORACLE_OK;
}

int gdn_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
