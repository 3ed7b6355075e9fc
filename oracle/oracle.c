/*
 * Oracle: a plain, slow, float64 CPU statement of what the hot path computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header, table or helper with the CUDA
 * library, and it is compiled without -ffast-math and with -ffp-contract=off
 * so that x86-64 and AArch64 hosts give the same bits.
 *
 * Sources (page "HDBSCAN", neuro-kitchen dsp-kitchen gpu/hdbscan, and page
 * "Kilosort4 clustering and matching", gpu/clustering):
 *
 *  - k-NN: each query's k nearest points of a set, by Euclidean distance
 *    (clustering page, section "k-nearest neighbours are a matrix product";
 *    the oracle sums the squared differences directly instead of expanding
 *    |x|^2 + |y|^2 - 2 x.y, which is the same quantity in exact arithmetic).
 *    Equal distances are ordered by ascending index of the set's column
 *    (hdbscan page, "The hang": the list keeps equal distances in scan order;
 *    "Exact shortcuts": lowest index wins).
 *  - Core distance: a point's distance to its min_samples-th nearest
 *    neighbour, the point itself included and counted first (hdbscan page,
 *    "The algorithm on the device").
 *  - Mutual-reachability weight max(core_a, core_b, |a - b|) and its minimum
 *    spanning tree with ties broken by (weight, lower index, higher index),
 *    which makes the tree unique (same section).  The page's upstream builds
 *    it with Prim's algorithm over every pair ("HDBSCAN", introduction); the
 *    oracle does the same, dense, O(n^2).
 *
 * Every function returns 0 on success and a negative value on bad arguments.
 * Inputs are float32, feature-major [d, n] with leading dimension ld >= n:
 * feature f of point i is X[f * ld + i].  Indices are int64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <omp.h>

int oracle_threads(void) { return omp_get_max_threads(); }

/* Copy a feature-major [d, n] float set into point-major rows of d floats.
 * A layout change only: values are copied unchanged. */
static float *to_point_major(const float *X, int64_t ld, int64_t n, int d) {
    float *P = (float *)malloc(sizeof(float) * (size_t)n * (size_t)d + 1);
    if (!P) return NULL;
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        for (int f = 0; f < d; ++f) P[i * d + f] = X[(int64_t)f * ld + i];
    return P;
}

/* Euclidean distance between two points of d float32 features, in float64:
 * the squared differences summed in ascending feature order, then sqrt. */
static double dist64(const float *a, const float *b, int d) {
    double s = 0.0;
    for (int f = 0; f < d; ++f) {
        double t = (double)a[f] - (double)b[f];
        s += t * t;
    }
    return sqrt(s);
}

/* (dist, index) lexicographic order. */
static int dj_less(double da, int64_t ja, double db, int64_t jb) {
    return da < db || (da == db && ja < jb);
}

/*
 * Exact k-NN: for every query column i of Xq [d, nq], the k columns j of Y
 * [d, m] with the smallest (dist(i, j), j).  Writes out_idx[i * k + r] and
 * out_dist[i * k + r] for r = 0 .. k-1 in that order.  Self matches are kept
 * when Y contains the query.
 */
int oracle_knn(const float *Xq, int64_t ldq, int64_t nq, const float *Y, int64_t ldy,
               int64_t m, int d, int k, int64_t *out_idx, double *out_dist) {
    if (nq < 0 || m < 1 || d < 1 || k < 1 || k > m || ldq < nq || ldy < m) return -1;
    float *Q = to_point_major(Xq, ldq, nq, d);
    float *P = to_point_major(Y, ldy, m, d);
    if (!Q || !P) { free(Q); free(P); return -2; }
    #pragma omp parallel
    {
        double *bd = (double *)malloc(sizeof(double) * (size_t)k);
        int64_t *bj = (int64_t *)malloc(sizeof(int64_t) * (size_t)k);
        #pragma omp for schedule(dynamic, 16)
        for (int64_t i = 0; i < nq; ++i) {
            int cnt = 0;
            for (int64_t j = 0; j < m; ++j) {
                double dj = dist64(Q + i * d, P + j * d, d);
                if (cnt == k && !dj_less(dj, j, bd[k - 1], bj[k - 1])) continue;
                /* insertion into the sorted list, dropping the last if full */
                int pos = cnt < k ? cnt : k - 1;
                while (pos > 0 && dj_less(dj, j, bd[pos - 1], bj[pos - 1])) {
                    bd[pos] = bd[pos - 1];
                    bj[pos] = bj[pos - 1];
                    --pos;
                }
                bd[pos] = dj;
                bj[pos] = j;
                if (cnt < k) ++cnt;
            }
            for (int r = 0; r < k; ++r) {
                out_idx[i * k + r] = bj[r];
                out_dist[i * k + r] = bd[r];
            }
        }
        free(bd);
        free(bj);
    }
    free(Q);
    free(P);
    return 0;
}

/*
 * Core distances: core_i is the distance from point i to its min_samples-th
 * nearest point of X, i itself included (so min_samples = 1 gives 0).
 * Rows Xq [d, nq] are the points whose core distance is wanted; X [d, n] is
 * the whole set (pass the same array twice for every point).
 */
int oracle_core_distances(const float *Xq, int64_t ldq, int64_t nq, const float *X,
                          int64_t ldx, int64_t n, int d, int min_samples, double *out_core) {
    if (min_samples < 1 || min_samples > n) return -1;
    int64_t *idx = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nq > 0 ? nq : 1) * min_samples);
    double *dist = (double *)malloc(sizeof(double) * (size_t)(nq > 0 ? nq : 1) * min_samples);
    if (!idx || !dist) { free(idx); free(dist); return -2; }
    int rc = oracle_knn(Xq, ldq, nq, X, ldx, n, d, min_samples, idx, dist);
    if (rc == 0)
        for (int64_t i = 0; i < nq; ++i) out_core[i] = dist[i * min_samples + (min_samples - 1)];
    free(idx);
    free(dist);
    return rc;
}

/* An edge key: (weight, lower index, higher index), compared lexicographically. */
typedef struct { double w; int64_t lo, hi; } okey;

static int key_less(const okey *a, const okey *b) {
    if (a->w != b->w) return a->w < b->w;
    if (a->lo != b->lo) return a->lo < b->lo;
    return a->hi < b->hi;
}

static okey mr_key(const float *P, const double *core, int64_t a, int64_t b, int d) {
    okey k;
    double w = dist64(P + a * d, P + b * d, d);
    if (core[a] > w) w = core[a];
    if (core[b] > w) w = core[b];
    k.w = w;
    k.lo = a < b ? a : b;
    k.hi = a < b ? b : a;
    return k;
}

static int key_cmp(const void *pa, const void *pb) {
    const okey *a = (const okey *)pa, *b = (const okey *)pb;
    if (key_less(a, b)) return -1;
    if (key_less(b, a)) return 1;
    return 0;
}

/*
 * Minimum spanning tree of the mutual-reachability weights by dense Prim:
 * grow a tree from point 0; every non-tree point keeps the least key of an
 * edge to the tree; each step moves the point with the least such key into
 * the tree and relaxes every remaining point against it.  Under the strict
 * (weight, lo, hi) order the tree is unique.
 *
 * core[n] is in float64.  Writes n-1 edges sorted by (w, lo, hi):
 * out_lo[e] < out_hi[e], out_w[e] the float64 weight.
 */
int oracle_prim_mst(const float *X, int64_t ldx, int64_t n, int d, const double *core,
                    int64_t *out_lo, int64_t *out_hi, double *out_w) {
    if (n < 1 || d < 1 || ldx < n) return -1;
    if (n == 1) return 0;
    float *P = to_point_major(X, ldx, n, d);
    okey *best = (okey *)malloc(sizeof(okey) * (size_t)n);
    int64_t *rem = (int64_t *)malloc(sizeof(int64_t) * (size_t)n);
    okey *edges = (okey *)malloc(sizeof(okey) * (size_t)n);
    int nt = omp_get_max_threads();
    int64_t *tmin = (int64_t *)malloc(sizeof(int64_t) * (size_t)nt);
    if (!P || !best || !rem || !edges || !tmin) {
        free(P); free(best); free(rem); free(edges); free(tmin);
        return -2;
    }
    /* the tree starts as {0}; rem lists the points outside it */
    int64_t nrem = n - 1;
    for (int64_t i = 0; i < nrem; ++i) rem[i] = i + 1;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrem; ++r) best[rem[r]] = mr_key(P, core, 0, rem[r], d);

    for (int64_t step = 0; step < n - 1; ++step) {
        /* position in rem of the least key: each thread scans a share, then
         * the shares are compared in a fixed order (keys are all distinct) */
        #pragma omp parallel
        {
            int t = omp_get_thread_num();
            int64_t bi = -1;
            #pragma omp for schedule(static)
            for (int64_t r = 0; r < nrem; ++r)
                if (bi < 0 || key_less(&best[rem[r]], &best[rem[bi]])) bi = r;
            tmin[t] = bi;
        }
        int64_t pos = -1;
        for (int t = 0; t < nt; ++t)
            if (tmin[t] >= 0 && (pos < 0 || key_less(&best[rem[tmin[t]]], &best[rem[pos]])))
                pos = tmin[t];
        int64_t v = rem[pos];
        edges[step] = best[v];
        rem[pos] = rem[nrem - 1];
        --nrem;
        #pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < nrem; ++r) {
            int64_t u = rem[r];
            okey kv = mr_key(P, core, v, u, d);
            if (key_less(&kv, &best[u])) best[u] = kv;
        }
    }
    qsort(edges, (size_t)(n - 1), sizeof(okey), key_cmp);
    for (int64_t e = 0; e < n - 1; ++e) {
        out_lo[e] = edges[e].lo;
        out_hi[e] = edges[e].hi;
        out_w[e] = edges[e].w;
    }
    free(P); free(best); free(rem); free(edges); free(tmin);
    return 0;
}

/* float64 Euclidean distance of listed pairs (a[e], b[e]) of X [d, n]. */
int oracle_pair_dist(const float *X, int64_t ldx, int64_t n, int d, const int64_t *a,
                     const int64_t *b, int64_t cnt, double *out) {
    if (n < 1 || d < 1 || ldx < n) return -1;
    for (int64_t e = 0; e < cnt; ++e)
        if (a[e] < 0 || a[e] >= n || b[e] < 0 || b[e] >= n) return -1;
    #pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < cnt; ++e) {
        double s = 0.0;
        for (int f = 0; f < d; ++f) {
            double t = (double)X[(int64_t)f * ldx + a[e]] - (double)X[(int64_t)f * ldx + b[e]];
            s += t * t;
        }
        out[e] = sqrt(s);
    }
    return 0;
}
