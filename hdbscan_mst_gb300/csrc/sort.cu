// K9: order the tree's edges by (w, lo, hi).
//
// The pages leave the output order open; (w, lo, hi) is the tree's own total
// order (the order Kruskal would add the edges in, which a single-linkage
// hierarchy consumes directly).  Edges come out of the Boruvka rounds in
// atomic-append order, so they are sorted here by a stable least-significant
// digit radix sort on 8-bit digits: the digits of hi, then lo, then the
// weight's bits (non-negative floats order like their bit patterns).
//
// One pass = per-tile digit histograms, then a stable scatter: each block
// sums the histograms into its tile's first position per digit (all smaller
// digits, then the same digit in earlier tiles) and each warp ranks equal
// digits with __match_any_sync.
#include "common.cuh"
#include "internal.h"

namespace hdbmst {

namespace {

constexpr int kSortThreads = 256;
constexpr int kSortRounds = 8;
constexpr int kSortTile = kSortThreads * kSortRounds;  // elements per block

__global__ void __launch_bounds__(kSortThreads) hist_kernel(int N, const unsigned *__restrict__ key,
                                                            int shift, unsigned *__restrict__ hist,
                                                            int tiles) {
    __shared__ unsigned h[256];
    h[threadIdx.x] = 0;
    __syncthreads();
    const int base = blockIdx.x * kSortTile;
    for (int q = 0; q < kSortRounds; ++q) {
        const int e = base + q * kSortThreads + threadIdx.x;
        if (e < N) atomicAdd(&h[(key[e] >> shift) & 255u], 1u);
    }
    __syncthreads();
    hist[threadIdx.x * tiles + blockIdx.x] = h[threadIdx.x];
}

__global__ void __launch_bounds__(kSortThreads) scatter_kernel(
    int N, int shift, int which, const unsigned *__restrict__ w, const int *__restrict__ lo,
    const int *__restrict__ hi, unsigned *__restrict__ w2, int *__restrict__ lo2,
    int *__restrict__ hi2, const unsigned *__restrict__ hist, int tiles) {
    __shared__ unsigned offset[256];
    __shared__ unsigned wcnt[kSortThreads / 32][256];
    __shared__ unsigned wsum[kSortThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    // This tile's first position for digit tid: the count of all smaller
    // digits plus that of digit tid in the tiles before this one.
    unsigned before = 0, total = 0;
    for (int t = 0; t < tiles; ++t) {
        const unsigned v = hist[tid * tiles + t];
        before += t < static_cast<int>(blockIdx.x) ? v : 0u;
        total += v;
    }
    unsigned incl = total;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[wid] = incl;
    for (int q = 0; q < kSortThreads / 32; ++q) wcnt[q][tid] = 0;
    __syncthreads();
    unsigned wbefore = 0;
    for (int q = 0; q < wid; ++q) wbefore += wsum[q];
    offset[tid] = wbefore + incl - total + before;
    __syncthreads();
    const int base = blockIdx.x * kSortTile;
    for (int q = 0; q < kSortRounds; ++q) {
        const int e = base + q * kSortThreads + tid;
        const bool valid = e < N;
        unsigned kw = 0, digit = 256u + lane;  // invalid lanes: a digit of their own
        int klo = 0, khi = 0;
        if (valid) {
            kw = w[e];
            klo = lo[e];
            khi = hi[e];
            const unsigned kk = which == 0 ? static_cast<unsigned>(khi)
                                : which == 1 ? static_cast<unsigned>(klo)
                                             : kw;
            digit = (kk >> shift) & 255u;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, digit);
        const unsigned rank = __popc(peers & lanemask_lt());
        if (valid && rank == 0) wcnt[wid][digit] = __popc(peers);
        __syncthreads();
        if (valid) {
            unsigned pos = offset[digit] + rank;
            for (int v = 0; v < wid; ++v) pos += wcnt[v][digit];
            w2[pos] = kw;
            lo2[pos] = klo;
            hi2[pos] = khi;
        }
        __syncthreads();
        unsigned tot = 0;
        for (int v = 0; v < kSortThreads / 32; ++v) {
            tot += wcnt[v][tid];
            wcnt[v][tid] = 0;
        }
        offset[tid] += tot;
        __syncthreads();
    }
}

__global__ void write_edges_kernel(int N, const unsigned *__restrict__ w, const int *__restrict__ lo,
                                   const int *__restrict__ hi, int32_t *__restrict__ out_edges,
                                   float *__restrict__ out_w) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= N) return;
    out_edges[2 * static_cast<int64_t>(e)] = lo[e];
    out_edges[2 * static_cast<int64_t>(e) + 1] = hi[e];
    out_w[e] = __uint_as_float(w[e]);
}

inline int tiles_for(int N) { return (N + kSortTile - 1) / kSortTile; }

}  // namespace

size_t sort_hist_entries(int N) { return static_cast<size_t>(256) * tiles_for(N > 0 ? N : 1); }

int sort_launches(int N, int index_bits) {
    const int ip = (index_bits + 7) / 8;
    return (2 * ip + 4) * 2 + 1;
}

cudaError_t sort_edges(int N, int index_bits, unsigned *w, int *lo, int *hi, unsigned *w2,
                       int *lo2, int *hi2, unsigned *hist, int32_t *out_edges, float *out_w,
                       cudaStream_t s, void (*before)(int, cudaStream_t),
                       void (*after)(int, cudaStream_t)) {
    if (N <= 0) return cudaSuccess;
    const int tiles = tiles_for(N);
    const int ip = (index_bits + 7) / 8;
    struct Pass { int which, shift; };
    Pass passes[12];
    int np = 0;
    for (int b = 0; b < ip; ++b) passes[np++] = {0, 8 * b};
    for (int b = 0; b < ip; ++b) passes[np++] = {1, 8 * b};
    for (int b = 0; b < 4; ++b) passes[np++] = {2, 8 * b};
    unsigned *sw = w, *dw = w2;
    int *slo = lo, *dlo = lo2, *shi = hi, *dhi = hi2;
    for (int p = 0; p < np; ++p) {
        const unsigned *key = passes[p].which == 0 ? reinterpret_cast<const unsigned *>(shi)
                              : passes[p].which == 1 ? reinterpret_cast<const unsigned *>(slo)
                                                     : sw;
        before(K_SORT, s);
        hist_kernel<<<tiles, kSortThreads, 0, s>>>(N, key, passes[p].shift, hist, tiles);
        after(K_SORT, s);
        before(K_SORT, s);
        scatter_kernel<<<tiles, kSortThreads, 0, s>>>(N, passes[p].shift, passes[p].which, sw, slo,
                                                      shi, dw, dlo, dhi, hist, tiles);
        after(K_SORT, s);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        unsigned *tw = sw; sw = dw; dw = tw;
        int *t1 = slo; slo = dlo; dlo = t1;
        int *t2 = shi; shi = dhi; dhi = t2;
    }
    before(K_SORT, s);
    write_edges_kernel<<<(N + 255) / 256, 256, 0, s>>>(N, sw, slo, shi, out_edges, out_w);
    after(K_SORT, s);
    return cudaGetLastError();
}

}  // namespace hdbmst
