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

// The pivots' features, feature-major [dp][P] (dp = d rounded up to 16, zero
// rows past d): pivot p is the column point p * stride of Y.
__global__ void pivots_kernel(const float *__restrict__ Y, int64_t ldy, int stride, int d, int dp,
                              int P, float *__restrict__ piv) {
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= dp * P) return;
    const int f = q / P, p = q % P;
    piv[q] = f < d ? Y[static_cast<int64_t>(f) * ldy + static_cast<int64_t>(p) * stride] : 0.f;
}

// Nearest pivot of each point of S (feature-major, leading dimension lds),
// ties to the lower pivot; also the point's distance to its own pivot
// (dcell), its distances to all 128 pivots if pd is not null (point-major
// [cnt][128]), cmax[cell] raised to the distance to its own pivot, and
// *amax_bits (if not null) to the largest finite magnitude in S.  A CTA
// of 256 threads takes 128 points against the 128 pivots; thread (ty, tx)
// accumulates points 8 ty .. 8 ty + 7 against pivots 4 tx .. 4 tx + 3 and
// 64 + 4 tx .. 64 + 4 tx + 3, so that the eight lanes of a quarter warp read
// 128 contiguous bytes of pivots from shared memory (one wavefront) and one
// broadcast word group of points.  Features go 16 at a time through shared
// memory; the next 16 are loaded into registers while these are used.  Each
// squared distance is the same ascending-feature chain of fused
// multiply-adds of differences as one point at a time would give.
constexpr int kCellPts = 128, kCellPiv = 128, kCellK = 16;
constexpr int kCellLoads = kCellK * kCellPts / 256;  // per thread and stage, for each operand
static_assert(kCellPts == kCellPiv, "one load pattern for points and pivots");

__global__ void __launch_bounds__(256, 2) cells_kernel(const float *__restrict__ S, int64_t lds,
                                                       int cnt, int d, const float *__restrict__ piv,
                                                       int dp, int *__restrict__ cell,
                                                       float *__restrict__ dcell,
                                                       float *__restrict__ pd,
                                                       unsigned *__restrict__ cmax,
                                                       unsigned *__restrict__ amax_bits) {
    __shared__ __align__(16) float xs[kCellK][kCellPts];
    __shared__ __align__(16) float ps[kCellK][kCellPiv];
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int i0 = blockIdx.x * kCellPts;
    // stage loads: element tid + 256 r of the [16][128] tile, r < kCellLoads
    const int lc = tid & (kCellPts - 1), lf = tid / kCellPts;
    float rx[kCellLoads], rp[kCellLoads];
    unsigned amax = 0u;  // the largest finite magnitude this thread loaded (as bits)
    const auto load_stage = [&](int f0) {
#pragma unroll
        for (int r = 0; r < kCellLoads; ++r) {
            const int f = f0 + lf + r * (256 / kCellPts);
            const int i = i0 + lc;
            rx[r] = (i < cnt && f < d) ? S[static_cast<int64_t>(f) * lds + i] : 0.f;
            // the pivots negated: x + (-p) rounds exactly as x - p
            rp[r] = -piv[static_cast<int64_t>(f) * kCellPiv + lc];
        }
#pragma unroll
        for (int r = 0; r < kCellLoads; ++r) {
            // non-negative floats order like their bits; non-finite values
            // are the pack kernel's to report
            const float v = fabsf(rx[r]);
            if (v <= 3.4028234663852886e38f) amax = max(amax, __float_as_uint(v));
        }
    };
    // acc[a][b]: point 8 ty + a against pivots 4 tx + 2 b, + 1 (b < 2) or
    // 64 + 4 tx + 2 (b - 2), + 1 (b >= 2): packed FP32 pairs, each half
    // summed in feature order exactly as a scalar FMA chain
    float2 acc[8][4];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = make_float2(0.f, 0.f);
    load_stage(0);
    for (int f0 = 0; f0 < dp; f0 += kCellK) {
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kCellLoads; ++r) {
            xs[lf + r * (256 / kCellPts)][lc] = rx[r];
            ps[lf + r * (256 / kCellPts)][lc] = rp[r];
        }
        __syncthreads();
        if (f0 + kCellK < dp) load_stage(f0 + kCellK);
#pragma unroll
        for (int f = 0; f < kCellK; ++f) {
            const float4 x0 = *reinterpret_cast<const float4 *>(&xs[f][ty * 8]);
            const float4 x1 = *reinterpret_cast<const float4 *>(&xs[f][ty * 8 + 4]);
            const float4 p0 = *reinterpret_cast<const float4 *>(&ps[f][tx * 4]);
            const float4 p1 = *reinterpret_cast<const float4 *>(&ps[f][64 + tx * 4]);
            const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            const float2 pv[4] = {make_float2(p0.x, p0.y), make_float2(p0.z, p0.w),
                                  make_float2(p1.x, p1.y), make_float2(p1.z, p1.w)};
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                const float2 x2 = make_float2(xv[a], xv[a]);
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const float2 t = __fadd2_rn(x2, pv[b]);
                    acc[a][b] = __ffma2_rn(t, t, acc[a][b]);
                }
            }
        }
    }
    if (amax_bits) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if ((tid & 31) == 0 && amax) atomicMax(amax_bits, amax);
    }
#pragma unroll
    for (int a = 0; a < 8; ++a) {
        const int i = i0 + ty * 8 + a;
        // the thread's pivots in ascending order
        const float sq[8] = {acc[a][0].x, acc[a][0].y, acc[a][1].x, acc[a][1].y,
                             acc[a][2].x, acc[a][2].y, acc[a][3].x, acc[a][3].y};
        float best = sq[0];
        int arg = tx * 4;
#pragma unroll
        for (int b = 1; b < 8; ++b)
            if (sq[b] < best) {
                best = sq[b];
                arg = (b < 4 ? 0 : 60) + tx * 4 + b;
            }
        // least (value, pivot) over the 16 lanes of this point (one half-warp)
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oa = __shfl_xor_sync(0xffffffffu, arg, o);
            if (ob < best || (ob == best && oa < arg)) {
                best = ob;
                arg = oa;
            }
        }
        if (i < cnt) {
            if (pd) {
                float *row = pd + static_cast<int64_t>(i) * kCellPiv;
                *reinterpret_cast<float4 *>(row + tx * 4) =
                    make_float4(__fsqrt_rn(sq[0]), __fsqrt_rn(sq[1]), __fsqrt_rn(sq[2]),
                                __fsqrt_rn(sq[3]));
                *reinterpret_cast<float4 *>(row + 64 + tx * 4) =
                    make_float4(__fsqrt_rn(sq[4]), __fsqrt_rn(sq[5]), __fsqrt_rn(sq[6]),
                                __fsqrt_rn(sq[7]));
            }
            if (tx == 0) {
                cell[i] = arg;
                const float dc = __fsqrt_rn(best);
                dcell[i] = dc;
                // non-negative floats order like their bits
                atomicMax(&cmax[arg], __float_as_uint(dc));
            }
        }
    }
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

// start[c] = points in bins before c, start[P] = all: one CTA of 1024
// threads, each summing a run of consecutive bins, then a block-wide scan of
// the runs' totals.
__global__ void __launch_bounds__(1024) start_cells_kernel(const int *__restrict__ count, int P,
                                                           int *__restrict__ start) {
    __shared__ int s_warp[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (P + 1023) / 1024;
    const int b0 = min(tid * per, P), b1 = min(b0 + per, P);
    int run = 0;
    for (int c = b0; c < b1; ++c) run += count[c];
    int incl = run;  // inclusive scan of the runs: within the warp, then over warps
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = s_warp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        s_warp[lane] = w;
    }
    __syncthreads();
    int acc = (warp ? s_warp[warp - 1] : 0) + incl - run;
    for (int c = b0; c < b1; ++c) {
        start[c] = acc;
        acc += count[c];
    }
    if (tid == 1023) start[P] = acc;
}

__global__ void scatter_cells_kernel(const int *__restrict__ cell, int cnt,
                                     const int *__restrict__ start, int *__restrict__ cursor,
                                     int *__restrict__ perm, int *__restrict__ inv) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < cnt) {
        const int c = cell[i];
        const int pos = start[c] + atomicAdd(&cursor[c], 1);
        perm[pos] = i;
        inv[i] = pos;
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
                                 cudaStream_t s, unsigned *amax_bits) {
    const int P = o.pivots, B = o.buckets, NB = P * B;
    if (P != kCellPiv || d > kSpatialMaxD) return cudaErrorInvalidValue;
    const int stride = m / P;
    const int dp = (d + kCellK - 1) / kCellK * kCellK;
    pivots_kernel<<<blocks_for(dp * P, 256), 256, 0, s>>>(Y, ldy, stride, d, dp, P, o.pivf);
    // counters: count and cursor of Y's bins (and of X's), the cells' largest
    // pivot distances of Y (and of X), zeroed
    cudaError_t e = cudaMemsetAsync(o.counters, 0, sizeof(int) * spatial_counter_ints(P, B), s);
    if (e != cudaSuccess) return e;
    int *countY = o.counters, *cursorY = o.counters + NB, *countX = o.counters + 2 * NB,
        *cursorX = o.counters + 3 * NB;
    unsigned *cmaxY = reinterpret_cast<unsigned *>(o.counters + 4 * NB), *cmaxX = cmaxY + P;
    cells_kernel<<<blocks_for(m, kCellPts), 256, 0, s>>>(Y, ldy, m, d, o.pivf, dp, o.cellY,
                                                         o.dcellY, o.pdY, cmaxY, amax_bits);
    bins_kernel<<<blocks_for(m, 256), 256, 0, s>>>(o.cellY, o.dcellY, cmaxY, B, m, countY);
    start_cells_kernel<<<1, 1024, 0, s>>>(countY, NB, o.startY);
    scatter_cells_kernel<<<blocks_for(m, 256), 256, 0, s>>>(o.cellY, m, o.startY, cursorY, o.permY,
                                                           o.invY);
    int extra = 5;  // pivots, cells, bins, start, scatter, tile start: 6 kernels, one counted by the caller
    if (!alias) {
        cells_kernel<<<blocks_for(n, kCellPts), 256, 0, s>>>(X, ldx, n, d, o.pivf, dp, o.cellX,
                                                             o.dcellX, o.pdX, cmaxX, amax_bits);
        bins_kernel<<<blocks_for(n, 256), 256, 0, s>>>(o.cellX, o.dcellX, cmaxX, B, n, countX);
        start_cells_kernel<<<1, 1024, 0, s>>>(countX, NB, o.startX);
        scatter_cells_kernel<<<blocks_for(n, 256), 256, 0, s>>>(o.cellX, n, o.startX, cursorX,
                                                               o.permX, o.invX);
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
