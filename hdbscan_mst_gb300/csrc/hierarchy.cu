// The HDBSCAN back half on the host: the single-linkage merge tree of the
// minimum spanning tree, its condensed tree for min_cluster_size, cluster
// stabilities, excess-of-mass selection and point labels.
//
// Page "HDBSCAN" (gpu/hdbscan), "The algorithm on the device": after the
// spanning tree, the hierarchy, its condensed tree and the excess-of-mass
// selection run on the host, in linear time; the upstream sorter runs
// scikit-learn's HDBSCAN, whose definitions this file states:
//  * edge i = (lo, hi, w), taken in (w, lo, hi) order, merges the component
//    of lo (first child) with that of hi (second child) into node n + i;
//  * the condensed tree is built breadth-first from the root, first child
//    before second: a split whose two sides both hold min_cluster_size points
//    makes two new clusters; a side below the size sheds its points (each an
//    entry of lambda = 1 / w, infinite for w = 0) and the other side carries
//    the cluster on;
//  * a cluster's stability is the sum over its entries, in the order they
//    were made, of (lambda - its birth lambda) x entry size, the root born at
//    0 (the order fixes the float rounding, and matches the oracle's);
//  * excess of mass, bottom-up: a cluster is kept when its stability is at
//    least the summed resolved stability of its child clusters, and then
//    replaces every kept cluster below it; the root is never kept;
//  * a point's label is its nearest kept ancestor, clusters numbered 0, 1, ...
//    by ascending smallest point index; -1 (noise) where there is none.
// Host code only; no CUDA calls.
#include <cmath>
#include <cstdint>
#include <limits>
#include <vector>

#include "../../include/hdbmst.h"

namespace {

struct MergeTree {
    int64_t n;
    std::vector<int64_t> first, second;  // children of node n + i
    std::vector<double> dist;
    std::vector<int64_t> size;           // of every node, 2n - 1
};

// Union-find over the 2n - 1 nodes; returns false if an edge closes a cycle.
bool single_linkage(int64_t n, const int32_t *edges, const float *w, MergeTree &T) {
    T.n = n;
    T.first.resize(n - 1);
    T.second.resize(n - 1);
    T.dist.resize(n - 1);
    T.size.assign(2 * n - 1, 1);
    std::vector<int64_t> parent(2 * n - 1);
    for (int64_t i = 0; i < 2 * n - 1; ++i) parent[i] = i;
    auto find = [&](int64_t x) {
        int64_t r = x;
        while (parent[r] != r) r = parent[r];
        while (parent[x] != r) {
            const int64_t nx = parent[x];
            parent[x] = r;
            x = nx;
        }
        return r;
    };
    for (int64_t i = 0; i < n - 1; ++i) {
        const int64_t lo = edges[2 * i], hi = edges[2 * i + 1];
        if (lo < 0 || hi < 0 || lo >= n || hi >= n) return false;
        const int64_t a = find(lo), b = find(hi);
        if (a == b) return false;
        const int64_t node = n + i;
        parent[a] = node;
        parent[b] = node;
        T.size[node] = T.size[a] + T.size[b];
        T.first[i] = a;
        T.second[i] = b;
        T.dist[i] = static_cast<double>(w[i]);
    }
    return true;
}

struct Condensed {
    std::vector<int64_t> parent, child, csize;  // child < n: a point; else a cluster label
    std::vector<double> lam;
    int64_t clusters = 0;                      // labels n .. n + clusters - 1
};

double lambda_of(double d) { return d > 0.0 ? 1.0 / d : std::numeric_limits<double>::infinity(); }

void condense(const MergeTree &T, int64_t mcs, Condensed &C) {
    const int64_t n = T.n;
    const int64_t root = 2 * n - 2;
    std::vector<int64_t> relabel(2 * n - 1, -1);
    relabel[root] = n;
    int64_t next_label = n + 1;
    std::vector<int64_t> queue{root}, sub;
    C.parent.reserve(2 * n);
    C.child.reserve(2 * n);
    C.csize.reserve(2 * n);
    C.lam.reserve(2 * n);
    auto push = [&](int64_t p, int64_t c, double l, int64_t s) {
        C.parent.push_back(p);
        C.child.push_back(c);
        C.lam.push_back(l);
        C.csize.push_back(s);
    };
    // the points of a subtree, breadth-first, as entries of parent me
    auto shed = [&](int64_t node, int64_t me, double l) {
        sub.clear();
        sub.push_back(node);
        for (size_t h = 0; h < sub.size(); ++h) {
            const int64_t x = sub[h];
            if (x < n) {
                push(me, x, l, 1);
            } else {
                sub.push_back(T.first[x - n]);
                sub.push_back(T.second[x - n]);
            }
        }
    };
    for (size_t h = 0; h < queue.size(); ++h) {
        const int64_t node = queue[h];
        if (node < n) continue;
        const int64_t a = T.first[node - n], b = T.second[node - n];
        const double l = lambda_of(T.dist[node - n]);
        const int64_t sa = T.size[a], sb = T.size[b], me = relabel[node];
        if (sa >= mcs && sb >= mcs) {
            relabel[a] = next_label++;
            push(me, relabel[a], l, sa);
            queue.push_back(a);
            relabel[b] = next_label++;
            push(me, relabel[b], l, sb);
            queue.push_back(b);
        } else if (sa < mcs && sb < mcs) {
            shed(a, me, l);
            shed(b, me, l);
        } else if (sa < mcs) {
            shed(a, me, l);
            relabel[b] = me;
            queue.push_back(b);
        } else {
            shed(b, me, l);
            relabel[a] = me;
            queue.push_back(a);
        }
    }
    C.clusters = next_label - n;
}

}  // namespace

extern "C" hdbmst_status hdbmst_hdbscan_labels(const int32_t *edges, const float *w, int64_t n,
                                               int min_cluster_size, int32_t *labels) {
    if (n < 0 || n > HDBMST_NMAX || min_cluster_size < 2) return HDBMST_ERR_ARG;
    if (n == 0) return HDBMST_OK;
    if (!labels || (n > 1 && (!edges || !w))) return HDBMST_ERR_ARG;
    if (n == 1) {
        labels[0] = -1;
        return HDBMST_OK;
    }
    for (int64_t i = 0; i < n - 1; ++i)
        if (!(w[i] >= 0.0f) || std::isinf(w[i])) return HDBMST_ERR_NONFINITE;
    MergeTree T;
    if (!single_linkage(n, edges, w, T)) return HDBMST_ERR_ARG;
    Condensed C;
    condense(T, min_cluster_size, C);
    const int64_t K = C.clusters;
    const size_t E = C.child.size();

    // stabilities, in entry order
    std::vector<double> birth(K, 0.0), stab(K, 0.0);
    for (size_t e = 0; e < E; ++e)
        if (C.child[e] >= n) birth[C.child[e] - n] = C.lam[e];
    for (size_t e = 0; e < E; ++e) {
        const int64_t p = C.parent[e] - n;
        stab[p] += (C.lam[e] - birth[p]) * static_cast<double>(C.csize[e]);
    }

    // child clusters of each cluster, in entry order (CSR)
    std::vector<int64_t> kid_start(K + 1, 0), kids;
    for (size_t e = 0; e < E; ++e)
        if (C.child[e] >= n) ++kid_start[C.parent[e] - n + 1];
    for (int64_t c = 0; c < K; ++c) kid_start[c + 1] += kid_start[c];
    kids.resize(kid_start[K]);
    {
        std::vector<int64_t> fill(kid_start.begin(), kid_start.end() - 1);
        for (size_t e = 0; e < E; ++e)
            if (C.child[e] >= n) kids[fill[C.parent[e] - n]++] = C.child[e] - n;
    }

    // excess of mass, children (larger labels) before parents; the root is
    // label 0 here and never a candidate
    std::vector<char> chosen(K, 0);
    std::vector<int64_t> stack;
    for (int64_t c = K - 1; c >= 1; --c) {
        double below = 0.0;
        for (int64_t q = kid_start[c]; q < kid_start[c + 1]; ++q) below += stab[kids[q]];
        if (below > stab[c]) {
            stab[c] = below;
        } else {
            chosen[c] = 1;
            stack.assign(kids.begin() + kid_start[c], kids.begin() + kid_start[c + 1]);
            while (!stack.empty()) {
                const int64_t x = stack.back();
                stack.pop_back();
                chosen[x] = 0;
                for (int64_t q = kid_start[x]; q < kid_start[x + 1]; ++q) stack.push_back(kids[q]);
            }
        }
    }

    // nearest chosen ancestor: clusters resolved top-down (a parent's label
    // is smaller than its children's), then each point through its entry
    std::vector<int64_t> up(K, -1), owner(K, -1);
    for (size_t e = 0; e < E; ++e)
        if (C.child[e] >= n) up[C.child[e] - n] = C.parent[e] - n;
    for (int64_t c = 0; c < K; ++c)
        owner[c] = chosen[c] ? c : (up[c] >= 0 ? owner[up[c]] : -1);
    std::vector<int64_t> point_owner(n, -1);
    for (size_t e = 0; e < E; ++e)
        if (C.child[e] < n) point_owner[C.child[e]] = owner[C.parent[e] - n];
    // clusters numbered by their smallest point index
    std::vector<int32_t> number(K, -1);
    int32_t next = 0;
    for (int64_t p = 0; p < n; ++p) {
        const int64_t c = point_owner[p];
        if (c >= 0 && number[c] < 0) number[c] = next++;
        labels[p] = c >= 0 ? number[c] : -1;
    }
    return HDBMST_OK;
}
