// K9: order the tree's edges by (w, lo, hi).
//
// The pages leave the output order open; (w, lo, hi) is the tree's own total
// order (the order Kruskal would add the edges in, which a single-linkage
// hierarchy consumes directly).  Edges come out of the Boruvka rounds in
// atomic-append order, so they are sorted here by a stable least-significant
// digit radix sort on 8-bit digits: the digits of hi, then lo, then the
// weight's bits (non-negative floats order like their bit patterns).
//
// A pass is one stable scatter over tiles of 2048 edges: each block sums the
// per-tile digit histograms into its tile's first position per digit (all
// smaller digits, then the same digit in earlier tiles) and each warp ranks
// equal digits with __match_any_sync.  The histograms of the next pass are
// counted by the scatter itself: every edge knows the tile it lands in and
// its next digit, and the lanes of a warp that share both add once.  Three
// histogram buffers rotate: pass p reads h[p % 3], counts into h[(p + 1) % 3]
// and clears h[(p + 2) % 3] for the pass after; only the first pass's
// histogram takes a launch of its own, and the last pass writes the output
// pairs and weights directly.
#include "common.cuh"
#include "internal.h"

namespace hdbmst {

namespace {

constexpr int kSortThreads = 256;
constexpr int kSortRounds = 8;
constexpr int kSortTile = kSortThreads * kSortRounds;  // elements per block

// which: 0 = hi, 1 = lo, 2 = the weight's bits
__device__ __forceinline__ unsigned digit_of(int which, int shift, unsigned w, int lo, int hi) {
    const unsigned k = which == 0 ? static_cast<unsigned>(hi)
                       : which == 1 ? static_cast<unsigned>(lo)
                                    : w;
    return (k >> shift) & 255u;
}

// The first pass's per-tile histograms (tile-major: hist[tile * 256 +
// digit]), and the buffer the first pass counts into cleared.
__global__ void __launch_bounds__(kSortThreads) hist_kernel(int N, const unsigned *__restrict__ key,
                                                            int shift, unsigned *__restrict__ hist,
                                                            unsigned *__restrict__ clear, int tiles) {
    __shared__ unsigned h[256];
    h[threadIdx.x] = 0;
    clear[blockIdx.x * 256 + threadIdx.x] = 0;
    __syncthreads();
    const int base = blockIdx.x * kSortTile;
    for (int q = 0; q < kSortRounds; ++q) {
        const int e = base + q * kSortThreads + threadIdx.x;
        if (e < N) atomicAdd(&h[(key[e] >> shift) & 255u], 1u);
    }
    __syncthreads();
    hist[blockIdx.x * 256 + threadIdx.x] = h[threadIdx.x];
}

struct SortPassArgs {
    int N, tiles;
    int which, shift;          // this pass's digit
    int nwhich, nshift;        // the next pass's digit; nwhich < 0: last pass
    const unsigned *w;
    const int *lo, *hi;
    unsigned *w2;              // destination (not the last pass)
    int *lo2, *hi2;
    const unsigned *hist;      // this pass's histograms
    unsigned *hist_next;       // the next pass's, counted here (zero on entry)
    unsigned *hist_clear;      // cleared here for the pass after next
    int32_t *out_edges;        // the last pass: (lo, hi) pairs and weights
    float *out_w;
};

__global__ void __launch_bounds__(kSortThreads) scatter_kernel(const SortPassArgs a) {
    __shared__ unsigned offset[256];
    __shared__ unsigned wcnt[kSortThreads / 32][256];
    __shared__ unsigned wsum[kSortThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const bool last = a.nwhich < 0;
    if (!last) a.hist_clear[blockIdx.x * 256 + tid] = 0;
    // This tile's first position for digit tid: the count of all smaller
    // digits plus that of digit tid in the tiles before this one (each step
    // over the tiles one coalesced row of 256 counts, several in flight)
    unsigned before = 0, total = 0;
#pragma unroll 32
    for (int t = 0; t < a.tiles; ++t) {
        const unsigned v = a.hist[t * 256 + tid];
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
    // each round's edge is loaded one round ahead
    unsigned nw = 0;
    int nlo = 0, nhi = 0;
    if (base + tid < a.N) {
        nw = a.w[base + tid];
        nlo = a.lo[base + tid];
        nhi = a.hi[base + tid];
    }
    for (int q = 0; q < kSortRounds; ++q) {
        const int e = base + q * kSortThreads + tid;
        const bool valid = e < a.N;
        const unsigned kw = nw;
        const int klo = nlo, khi = nhi;
        if (q + 1 < kSortRounds && e + kSortThreads < a.N) {
            nw = a.w[e + kSortThreads];
            nlo = a.lo[e + kSortThreads];
            nhi = a.hi[e + kSortThreads];
        }
        unsigned digit = 256u + lane;  // invalid lanes: a digit of their own
        if (valid) digit = digit_of(a.which, a.shift, kw, klo, khi);
        const unsigned peers = __match_any_sync(0xffffffffu, digit);
        const unsigned rank = __popc(peers & lanemask_lt());
        if (valid && rank == 0) wcnt[wid][digit] = __popc(peers);
        __syncthreads();
        unsigned pos = 0;
        if (valid) {
            pos = offset[digit] + rank;
            for (int v = 0; v < wid; ++v) pos += wcnt[v][digit];
            if (last) {
                a.out_edges[2 * static_cast<int64_t>(pos)] = klo;
                a.out_edges[2 * static_cast<int64_t>(pos) + 1] = khi;
                a.out_w[pos] = __uint_as_float(kw);
            } else {
                a.w2[pos] = kw;
                a.lo2[pos] = klo;
                a.hi2[pos] = khi;
            }
        }
        if (!last) {
            // the next pass's histogram: (next digit, destination tile), one
            // add per distinct pair in the warp
            const unsigned nd = valid ? digit_of(a.nwhich, a.nshift, kw, klo, khi) : 0u;
            const unsigned bin = valid ? (pos / kSortTile) * 256u + nd
                                       : 0xffffffffu - lane;  // invalid lanes alone
            const unsigned same = __match_any_sync(0xffffffffu, bin);
            if (valid && __popc(same & lanemask_lt()) == 0) atomicAdd(a.hist_next + bin, __popc(same));
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

inline int tiles_for(int N) { return (N + kSortTile - 1) / kSortTile; }

}  // namespace

size_t sort_hist_entries(int N) { return static_cast<size_t>(3) * 256 * tiles_for(N > 0 ? N : 1); }

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
    const size_t hsz = static_cast<size_t>(256) * tiles;
    unsigned *h[3] = {hist, hist + hsz, hist + 2 * hsz};
    before(K_SORT, s);
    hist_kernel<<<tiles, kSortThreads, 0, s>>>(N, reinterpret_cast<const unsigned *>(hi),
                                               passes[0].shift, h[0], h[1], tiles);
    after(K_SORT, s);
    unsigned *sw = w, *dw = w2;
    int *slo = lo, *dlo = lo2, *shi = hi, *dhi = hi2;
    for (int p = 0; p < np; ++p) {
        SortPassArgs a;
        a.N = N;
        a.tiles = tiles;
        a.which = passes[p].which;
        a.shift = passes[p].shift;
        a.nwhich = p + 1 < np ? passes[p + 1].which : -1;
        a.nshift = p + 1 < np ? passes[p + 1].shift : 0;
        a.w = sw;
        a.lo = slo;
        a.hi = shi;
        a.w2 = dw;
        a.lo2 = dlo;
        a.hi2 = dhi;
        a.hist = h[p % 3];
        a.hist_next = h[(p + 1) % 3];
        a.hist_clear = h[(p + 2) % 3];
        a.out_edges = out_edges;
        a.out_w = out_w;
        before(K_SORT, s);
        scatter_kernel<<<tiles, kSortThreads, 0, s>>>(a);
        after(K_SORT, s);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        unsigned *tw = sw; sw = dw; dw = tw;
        int *t1 = slo; slo = dlo; dlo = t1;
        int *t2 = shi; shi = dhi; dhi = t2;
    }
    return cudaSuccess;
}

}  // namespace hdbmst
