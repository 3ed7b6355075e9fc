// The k-NN graph consumer: bipartite modularity assignment (page "Kilosort4
// clustering and matching", gpu/clustering, section "Assignment in parallel:
// why the graph is bipartite").
//
// The graph joins every spike (a left node) to the k subset points (right
// nodes) its k-NN list names.  With the right labels fixed, a spike's best
// cluster depends on its own neighbours alone, so every spike is assigned at
// once (one thread each, its k neighbour labels in registers); then every
// subset point given the spikes' labels (every edge adds 1 to counts[r, c]
// with a 32-bit atomic, then one warp per subset point takes the best
// cluster); alternately.  A node takes, among its neighbours' labels, the c
// of largest 2m n_vc - gamma (k_v K_c): n_vc its edges to nodes labelled c,
// k_v its degree, K_c the degree sum of the other side's nodes labelled c,
// 2m twice the edge count; in float64 with the product of integers exact,
// gamma times it rounded once and the difference rounded once (explicit
// round-to-nearest intrinsics, so no multiply-add contraction); equal scores
// go to the lowest label.  The host reads one counter per round, the spikes
// the left step moved.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace hdbmst {

namespace {

__device__ __forceinline__ double assign_score(long long two_m, int n_vc, long long k_v,
                                               long long K_c, double gamma) {
    const double a = static_cast<double>(two_m * n_vc);
    const double b = __dmul_rn(gamma, static_cast<double>(k_v * K_c));
    return __dsub_rn(a, b);
}

// Right degrees (edges per subset point) and index checks; spikes start
// unlabelled (-1), so the first left step counts every spike as moved.
__global__ void assign_degree_kernel(const int32_t *__restrict__ nbr, int64_t edges, int k, int m,
                                     int *__restrict__ deg_r, int32_t *__restrict__ left,
                                     unsigned *__restrict__ status) {
    const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= edges) return;
    const int r = nbr[e];
    if (r < 0 || r >= m)
        atomicOr(status, kStatusBadList);
    else
        atomicAdd(&deg_r[r], 1);
    if (e % k == 0) left[e / k] = -1;
}

// K_c of the subset points (their degrees) for the left step; label checks.
__global__ void assign_right_mass_kernel(const int32_t *__restrict__ right, int m, int C,
                                         const int *__restrict__ deg_r,
                                         unsigned long long *__restrict__ K,
                                         unsigned *__restrict__ status) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= m) return;
    const int c = right[r];
    if (c < 0 || c >= C) {
        atomicOr(status, kStatusBadList);
        return;
    }
    if (deg_r[r]) atomicAdd(&K[c], static_cast<unsigned long long>(deg_r[r]));
}

// Left step: one thread per spike.  Writes the spike's new label, counts the
// spikes that moved (one atomic per warp) and adds the spike's degree k to
// the left mass of its new cluster (one atomic per warp and cluster).
template <int KM>
__global__ void __launch_bounds__(256) assign_left_kernel(
    const int32_t *__restrict__ nbr, int n, int k, int C, const int32_t *__restrict__ right,
    const unsigned long long *__restrict__ KR, double gamma, int32_t *__restrict__ left,
    unsigned long long *__restrict__ KL, int *__restrict__ moved) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const bool in = t < n;
    const long long two_m = 2ll * n * k;
    int lab[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        lab[j] = (in && j < k) ? right[nbr[static_cast<int64_t>(t) * k + j]] : INT_MAX;
        if (lab[j] < 0 || lab[j] >= C) lab[j] = INT_MAX;  // checked by the host first
    }
    int best = INT_MAX;
    double bs = -INFINITY;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        if (j < k && in && lab[j] != INT_MAX) {
            int cnt = 0;
#pragma unroll
            for (int i = 0; i < KM; ++i) cnt += (lab[i] == lab[j]) ? 1 : 0;
            const double sc = assign_score(two_m, cnt, k, static_cast<long long>(KR[lab[j]]), gamma);
            if (sc > bs || (sc == bs && lab[j] < best)) {
                bs = sc;
                best = lab[j];
            }
        }
    }
    const bool ok = in && best != INT_MAX;
    bool mv = false;
    if (ok) {
        mv = left[t] != best;
        left[t] = best;
    }
    const unsigned ball = __ballot_sync(0xffffffffu, mv);
    const int lane = threadIdx.x & 31;
    if (lane == 0 && ball) atomicAdd(moved, __popc(ball));
    const int key = ok ? best : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    if (ok && lane == __ffs(peers) - 1)
        atomicAdd(&KL[best], static_cast<unsigned long long>(__popc(peers)) * k);
}

// Right step, part 1: every edge (t, r) adds 1 to counts[r, label(t)].
__global__ void assign_count_kernel(const int32_t *__restrict__ nbr, int64_t edges, int k, int C,
                                    const int32_t *__restrict__ left,
                                    unsigned *__restrict__ counts) {
    const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= edges) return;
    atomicAdd(&counts[static_cast<int64_t>(nbr[e]) * C + left[e / k]], 1u);
}

// Right step, part 2: one warp per subset point; lanes read its counts row
// (coalesced), score the clusters it has edges to, and reduce to the best
// (largest score, then lowest label).  A point without edges keeps its label.
__global__ void __launch_bounds__(256) assign_right_kernel(
    const unsigned *__restrict__ counts, int m, int C, long long two_m,
    const int *__restrict__ deg_r, const unsigned long long *__restrict__ KL, double gamma,
    int32_t *__restrict__ right) {
    const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= m) return;  // whole warps
    const int dr = deg_r[r];
    if (dr == 0) return;
    const unsigned *row = counts + static_cast<int64_t>(r) * C;
    double bs = -INFINITY;
    int best = INT_MAX;
    for (int c = lane; c < C; c += 32) {
        const unsigned cnt = row[c];
        if (cnt == 0) continue;
        const double sc = assign_score(two_m, static_cast<int>(cnt), dr,
                                       static_cast<long long>(KL[c]), gamma);
        if (sc > bs) {  // ascending c per lane: the first maximum is the lowest label
            bs = sc;
            best = c;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const double os = __shfl_xor_sync(0xffffffffu, bs, o);
        const int ob = __shfl_xor_sync(0xffffffffu, best, o);
        if (os > bs || (os == bs && ob < best)) {
            bs = os;
            best = ob;
        }
    }
    if (lane == 0) right[r] = best;
}

inline int blocks_for(int64_t n, int t) { return static_cast<int>((n + t - 1) / t); }

}  // namespace

cudaError_t launch_assign_degree(const int32_t *nbr, int n, int k, int m, int *deg_r,
                                 int32_t *left, unsigned *status, cudaStream_t s) {
    const int64_t edges = static_cast<int64_t>(n) * k;
    if (edges == 0) return cudaSuccess;
    assign_degree_kernel<<<blocks_for(edges, 256), 256, 0, s>>>(nbr, edges, k, m, deg_r, left,
                                                                status);
    return cudaGetLastError();
}

cudaError_t launch_assign_right_mass(const int32_t *right, int m, int C, const int *deg_r,
                                     unsigned long long *KR, unsigned *status, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(KR, 0, sizeof(unsigned long long) * C, s);
    if (e != cudaSuccess || m == 0) return e;
    assign_right_mass_kernel<<<blocks_for(m, 256), 256, 0, s>>>(right, m, C, deg_r, KR, status);
    return cudaGetLastError();
}

cudaError_t launch_assign_left(const int32_t *nbr, int n, int k, int C, const int32_t *right,
                               const unsigned long long *KR, double gamma, int32_t *left,
                               unsigned long long *KL, int *moved, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(KL, 0, sizeof(unsigned long long) * C, s);
    if (e != cudaSuccess || n == 0) return e;
    if (k <= 16)
        assign_left_kernel<16><<<blocks_for(n, 256), 256, 0, s>>>(nbr, n, k, C, right, KR, gamma,
                                                                  left, KL, moved);
    else
        assign_left_kernel<32><<<blocks_for(n, 256), 256, 0, s>>>(nbr, n, k, C, right, KR, gamma,
                                                                  left, KL, moved);
    return cudaGetLastError();
}

cudaError_t launch_assign_right(const int32_t *nbr, int n, int k, int m, int C,
                                const int32_t *left, const int *deg_r,
                                const unsigned long long *KL, double gamma, unsigned *counts,
                                int32_t *right, cudaStream_t s) {
    const int64_t edges = static_cast<int64_t>(n) * k;
    cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(unsigned) * static_cast<size_t>(m) * C, s);
    if (e != cudaSuccess) return e;
    if (edges > 0) {
        assign_count_kernel<<<blocks_for(edges, 256), 256, 0, s>>>(nbr, edges, k, C, left,
                                                                   counts);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        count_extra_launches(1);
    }
    assign_right_kernel<<<blocks_for(static_cast<int64_t>(m) * 32, 256), 256, 0, s>>>(
        counts, m, C, 2ll * n * k, deg_r, KL, gamma, right);
    return cudaGetLastError();
}

}  // namespace hdbmst
