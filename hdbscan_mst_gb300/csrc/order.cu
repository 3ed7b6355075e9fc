// A spatial order for the tensor-core k-NN tile.
//
// The tile keeps, per row, the best candidates seen so far and filters every
// 32-column batch against the row's current threshold; batches with a
// candidate below it take the slow insertion path.  In the callers' order the
// columns of a row's neighbourhood are scattered over the whole sweep, and the
// threshold tightens only slowly.  Here every point goes to its nearest of P
// pivots (points of the column set at a fixed stride), rows and columns are
// sorted by pivot (counting sort), and each CTA starts its sweep at the block
// of columns of its first row's pivot: the first tiles it sees hold its rows'
// near neighbours, and the thresholds are nearly final after them.  The order
// changes which candidates are examined first, never the result: the refine
// maps positions back to the callers' indices before it ranks and proves.
//
// Within a cell the points are ordered by their distance to the pivot, in B
// buckets between 0 and the cell's largest distance: the far members of a
// cell (outliers that happen to lie nearest this pivot) then fill blocks of
// their own instead of widening every block of the cell, which is what lets
// the pruning of the column blocks (prune.cu) bound a block by the distances
// of its points to the pivots.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace hdbmst {

namespace {

int blocks_for(int n, int per) { return std::max(1, (n + per - 1) / per); }

// Nearest pivot of each point of S (feature-major, leading dimension lds):
// pivots in shared memory, 32 at a time per thread, ties to the lower pivot.
// Also writes the point's distance to its own pivot (dcell), its distances to
// all P pivots if pd is not null (point-major [cnt][P]), and raises cmax[cell]
// to its distance to its own pivot.
__global__ void __launch_bounds__(256) cells_kernel(const float *__restrict__ S, int64_t lds,
                                                    int cnt, const float *__restrict__ Y,
                                                    int64_t ldy, int stride, int d, int P,
                                                    int *__restrict__ cell,
                                                    float *__restrict__ dcell,
                                                    float *__restrict__ pd,
                                                    unsigned *__restrict__ cmax) {
    extern __shared__ float piv[];  // [P][d]
    for (int q = threadIdx.x; q < P * d; q += blockDim.x) {
        const int p = q / d, f = q % d;
        piv[q] = Y[static_cast<int64_t>(f) * ldy + static_cast<int64_t>(p) * stride];
    }
    __syncthreads();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= cnt) return;
    float best = INFINITY;
    int arg = 0;
    for (int c = 0; c < P; c += 32) {
        float acc[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) acc[q] = 0.f;
        for (int f = 0; f < d; ++f) {
            const float x = S[static_cast<int64_t>(f) * lds + i];
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const float t = x - piv[(c + q) * d + f];
                acc[q] = __fmaf_rn(t, t, acc[q]);
            }
        }
#pragma unroll
        for (int q = 0; q < 32; ++q)
            if (acc[q] < best) {
                best = acc[q];
                arg = c + q;
            }
        if (pd) {  // the point's distances to these 32 pivots (its point-major row of P)
            float4 *o = reinterpret_cast<float4 *>(pd + static_cast<int64_t>(i) * P + c);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                o[q] = make_float4(__fsqrt_rn(acc[4 * q]), __fsqrt_rn(acc[4 * q + 1]),
                                   __fsqrt_rn(acc[4 * q + 2]), __fsqrt_rn(acc[4 * q + 3]));
        }
    }
    cell[i] = arg;
    const float dc = __fsqrt_rn(best);
    dcell[i] = dc;
    // non-negative floats order like their bits
    atomicMax(&cmax[arg], __float_as_uint(dc));
}

// Bin of each point: its cell's bucket of distance to the pivot (B buckets
// between 0 and the cell's largest distance), bin = cell * B + bucket; the
// cell array is overwritten with the bin, and the bins are counted.
__global__ void bins_kernel(int *__restrict__ cell, const float *__restrict__ dcell,
                            const unsigned *__restrict__ cmax, int B, int cnt,
                            int *__restrict__ count) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= cnt) return;
    const int c = cell[i];
    const float mx = __uint_as_float(cmax[c]);
    const float dc = dcell[i];
    int q = 0;
    if (mx > 0.f) q = min(B - 1, max(0, static_cast<int>(dc / mx * static_cast<float>(B))));
    const int bin = c * B + q;
    cell[i] = bin;
    atomicAdd(&count[bin], 1);
}

// start[c] = points in bins before c (one warp), start[P] = all
__global__ void start_cells_kernel(const int *__restrict__ count, int P, int *__restrict__ start) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int b = 0; b < P; b += 32) {
        const int c = b + lane;
        const int v = c < P ? count[c] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (c < P) start[c] = carry + incl - v;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) start[P] = carry;
}

__global__ void scatter_cells_kernel(const int *__restrict__ cell, int cnt,
                                     const int *__restrict__ start, int *__restrict__ cursor,
                                     int *__restrict__ perm) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < cnt) {
        const int c = cell[i];
        perm[start[c] + atomicAdd(&cursor[c], 1)] = i;
    }
}

// Block (of 128 columns) where each row tile's sweep starts: the first block
// of the column cell of the tile's first row (binX holds bins of B buckets).
__global__ void tile_start_kernel(const int *__restrict__ permX, const int *__restrict__ binX,
                                  const int *__restrict__ startY, int B, int n, int row_tiles,
                                  int *__restrict__ tile_start) {
    const int rt = blockIdx.x * blockDim.x + threadIdx.x;
    if (rt >= row_tiles) return;
    const int r = min(rt * kBM, n - 1);
    tile_start[rt] = startY[binX[permX[r]] / B * B] / kBN;
}

}  // namespace

cudaError_t launch_spatial_order(const SpatialOrder &o, const float *X, int64_t ldx, int n,
                                 const float *Y, int64_t ldy, int m, bool alias, int d,
                                 cudaStream_t s) {
    const int P = o.pivots, B = o.buckets, NB = P * B;
    const int stride = m / P;
    const size_t smem = static_cast<size_t>(P) * d * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(cells_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // counters: count and cursor of Y's bins (and of X's), the cells' largest
    // pivot distances of Y (and of X), zeroed
    e = cudaMemsetAsync(o.counters, 0, sizeof(int) * spatial_counter_ints(P, B), s);
    if (e != cudaSuccess) return e;
    int *countY = o.counters, *cursorY = o.counters + NB, *countX = o.counters + 2 * NB,
        *cursorX = o.counters + 3 * NB;
    unsigned *cmaxY = reinterpret_cast<unsigned *>(o.counters + 4 * NB), *cmaxX = cmaxY + P;
    cells_kernel<<<blocks_for(m, 256), 256, smem, s>>>(Y, ldy, m, Y, ldy, stride, d, P, o.cellY,
                                                       o.dcellY, o.pdY, cmaxY);
    bins_kernel<<<blocks_for(m, 256), 256, 0, s>>>(o.cellY, o.dcellY, cmaxY, B, m, countY);
    start_cells_kernel<<<1, 32, 0, s>>>(countY, NB, o.startY);
    scatter_cells_kernel<<<blocks_for(m, 256), 256, 0, s>>>(o.cellY, m, o.startY, cursorY, o.permY);
    int extra = 4;  // cells, bins, start, scatter, tile start: 5 kernels, one counted by the caller
    if (!alias) {
        cells_kernel<<<blocks_for(n, 256), 256, smem, s>>>(X, ldx, n, Y, ldy, stride, d, P,
                                                           o.cellX, o.dcellX, o.pdX, cmaxX);
        bins_kernel<<<blocks_for(n, 256), 256, 0, s>>>(o.cellX, o.dcellX, cmaxX, B, n, countX);
        start_cells_kernel<<<1, 32, 0, s>>>(countX, NB, o.startX);
        scatter_cells_kernel<<<blocks_for(n, 256), 256, 0, s>>>(o.cellX, n, o.startX, cursorX,
                                                               o.permX);
        extra += 4;
    }
    const int row_tiles = (n + kBM - 1) / kBM;
    tile_start_kernel<<<blocks_for(row_tiles, 256), 256, 0, s>>>(
        alias ? o.permY : o.permX, alias ? o.cellY : o.cellX, o.startY, B, n, row_tiles,
        o.tile_start);
    count_extra_launches(extra);
    return cudaGetLastError();
}

}  // namespace hdbmst
