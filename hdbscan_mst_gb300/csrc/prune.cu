// Pruned column blocks for the tensor-core k-NN (exact).
//
// The page "Kilosort4 clustering and matching" (gpu/clustering, "k-nearest
// neighbours are a matrix product") computes every row against every column;
// the page "HDBSCAN" ("Exact shortcuts") skips work only where a bound proves
// it cannot change the result.  This file applies that rule to the distance
// tile: a 128-column block is skipped for a 128-row tile when the triangle
// inequality through one pivot of the spatial order (order.cu) proves that
// none of its points lies within any of the tile's rows' k-th distance.
//
// For a pivot p, a row x and a column z, |d(x, p) - d(z, p)| <= d(x, z).  A
// block whose points all have d(z, p) in [L, H] is therefore at least
// max(d(x, p) - H, L - d(x, p)) from x.  With an upper bound ub(x) of x's
// k-th distance, the block is useless to the tile if, for one pivot p,
// H < min over rows (d(x, p) - ub(x)) or L > max over rows (d(x, p) + ub(x)).
//
// The search runs in two passes of the tile.  The first ("home") pass takes
// a few blocks (home_blocks) around the columns of the tile's own bin; from its
// sorted candidates each row gets ub(x), a rigorous bound of the float32
// distance the refine will rank by (below).  The row tile's hull per pivot
// then selects the blocks of the second pass, which starts with the home
// pass's KP-th key as its rows' threshold.  The refine merges both passes and
// proves every row as before: a column the tile never evaluated lies, by the
// construction of ub, strictly beyond the refined k-th distance.
//
// Rounding.  Pivot distances are float32 direct differences, within relative
// eps = (d + 8) 2^-24 of the true ones (d + 2 roundings of the squared sum,
// one of the square root), and every bound is widened outward by eps.  ub(x)
// bounds the true distance of each of the k best home candidates by
// |x|^2 + t + c (|x|^2 + |y|^2) (c: the tile's ranking error bound), and is
// then scaled so that it also covers the float32 evaluation of the refine's
// distance, its strict-ordering margin and the rounding of this sum.
#include <cfloat>
#include <climits>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace hdbmst {

namespace {

constexpr int P = kPrunePivots;

int blocks_for(int64_t n, int per) { return static_cast<int>(n > per ? (n + per - 1) / per : 1); }

// Per column block b (one CTA, thread = pivot): least and largest distance of
// its points to the pivot, widened outward by eps; +inf / -inf for a block
// without points; pivot-major (Lm, Hm) and block-major (HLt) copies.  The
// pivot distances are in the callers' order (pdY[j][P]); a block holds the
// points permY[pos] of its sorted positions.  bcell[b]: the pivot cell of
// the block's first point.
__global__ void __launch_bounds__(P) block_bounds_kernel(const float *__restrict__ pdY, int m,
                                                         int col_tiles, double eps,
                                                         const int *__restrict__ binY,
                                                         const int *__restrict__ permY, int B,
                                                         float *__restrict__ Lm,
                                                         float *__restrict__ Hm,
                                                         float2 *__restrict__ HLt,
                                                         int *__restrict__ bcell) {
    static_assert(kBN == P, "one position per thread");
    __shared__ int s_pt[kBN];
    const int b = blockIdx.x, p = threadIdx.x;
    const int pos0 = b * kBN, pos1 = min(pos0 + kBN, m);
    s_pt[p] = pos0 + p < pos1 ? permY[pos0 + p] : 0;
    __syncthreads();
    float lo = INFINITY, hi = -INFINITY;
#pragma unroll 8
    for (int q = 0; q < pos1 - pos0; ++q) {
        const float v = pdY[static_cast<int64_t>(s_pt[q]) * P + p];
        lo = fminf(lo, v);
        hi = fmaxf(hi, v);
    }
    const int64_t o = static_cast<int64_t>(p) * col_tiles + b;
    const float L = pos1 > pos0 ? __double2float_rd(static_cast<double>(lo) * (1.0 - eps)) : INFINITY;
    const float H = pos1 > pos0 ? __double2float_ru(static_cast<double>(hi) * (1.0 + eps)) : -INFINITY;
    Lm[o] = L;
    Hm[o] = H;
    HLt[static_cast<int64_t>(b) * P + p] = make_float2(H, L);
    if (p == 0) bcell[b] = pos1 > pos0 ? binY[permY[pos0]] / B : 0;
}

// Per pivot (one CTA each): the least H and the largest L over all blocks.
__global__ void __launch_bounds__(256) pivot_range_kernel(const float *__restrict__ Lm,
                                                          const float *__restrict__ Hm,
                                                          int col_tiles, float *__restrict__ minH,
                                                          float *__restrict__ maxL) {
    __shared__ float s_h[8], s_l[8];
    const int p = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float h = INFINITY, l = -INFINITY;
    for (int b = tid; b < col_tiles; b += 256) {
        h = fminf(h, Hm[static_cast<int64_t>(p) * col_tiles + b]);
        l = fmaxf(l, Lm[static_cast<int64_t>(p) * col_tiles + b]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        h = fminf(h, __shfl_xor_sync(0xffffffffu, h, o));
        l = fmaxf(l, __shfl_xor_sync(0xffffffffu, l, o));
    }
    if (lane == 0) {
        s_h[warp] = h;
        s_l[warp] = l;
    }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < 8; ++w) {
            h = fminf(h, s_h[w]);
            l = fmaxf(l, s_l[w]);
        }
        minH[p] = h;
        maxL[p] = l;
    }
}

// Home range of each row tile of the chunk: nh blocks centred on the
// block that holds, in the columns' sorted order, the position matching the
// tile's middle row (its bin, at the same relative rank).  When Y is X that
// block holds the tile's own rows.
__global__ void home_kernel(const int *__restrict__ binX, const int *__restrict__ permX,
                            const int *__restrict__ startX, const int *__restrict__ startY,
                            int n, int col_tiles, int row_tile0, int row_tiles, int nh,
                            bool alias, int *__restrict__ home_lo, int *__restrict__ home) {
    const int rt = blockIdx.x * blockDim.x + threadIdx.x;
    if (rt >= row_tiles) return;
    const int gt = row_tile0 + rt;
    int hb;
    if (alias) {
        hb = gt;
    } else {
        const int q = min(gt * kBM + kBM / 2, n - 1);
        const int bin = binX[permX[q]];
        const int64_t rank = q - startX[bin];
        const int64_t cx = startX[bin + 1] - startX[bin];
        const int64_t cy = startY[bin + 1] - startY[bin];
        const int64_t pos = startY[bin] + (cy > 0 ? min(cy - 1, rank * cy / (cx > 0 ? cx : 1)) : 0);
        hb = static_cast<int>(pos / kBN);
    }
    const int h0 = max(0, min(hb - nh / 2, col_tiles - nh));
    home_lo[rt] = h0;
    for (int i = 0; i < nh; ++i) home[rt * kHomeBlocks + i] = h0 + i;
}

// One CTA (128 threads) per row tile of the chunk.
__global__ void __launch_bounds__(kBM, 12) prune_lists_kernel(const PruneListArgs a,
                                                          const float *__restrict__ Lm,
                                                          const float *__restrict__ Hm,
                                                          const float2 *__restrict__ HLt,
                                                          const int *__restrict__ bcell,
                                                          const int *__restrict__ home_lo,
                                                          int *__restrict__ list,
                                                          int *__restrict__ count,
                                                          int *__restrict__ slabs,
                                                          unsigned *__restrict__ b_gthr,
                                                          const float *__restrict__ minH,
                                                          const float *__restrict__ maxL) {
    __shared__ float s_ub[kBM];
    __shared__ float s_A[P], s_B[P];
    __shared__ int s_wc[kBM / 32];
    __shared__ int s_useful[P], s_nuseful;
    __shared__ int s_cand[kBM];
    __shared__ int s_keep[kBM];
    __shared__ int s_prow[kBM];  // the tile's points in the callers' order
    __shared__ unsigned long long s_near[kBM / 32];
    __shared__ float2 s_ABu[P];
    const int rt = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int local = rt * kBM + tid;
    const int row = a.row_base + local;
    const int nh = a.nh;

    // 1. ub(x) from the k best candidates of the home pass (sorted by (t, j)).
    //    True squared distance of candidate j: at most |x|^2 + t_j + c (|x|^2 +
    //    |y_j|^2) + e0 (the 1.01 covers the computed norms; e0 the FP16
    //    operands' absolute part).  The refine ranks by
    //    the float32 distance; its k-th value squared is at most (1 + (d + 5) u)
    //    times the largest of these, and a column is provably beyond it when
    //    its true squared distance exceeds that times (1 + 16 u) / (1 - (d + 3) u)
    //    (the refine's own margin).  The scale (1 + (4 d + 64) u) covers both
    //    with room for the rounding of this sum.
    float ub = -1.f;  // < 0: no row here
    if (row < a.row_end) {
        const float xn = a.xnorm[row], e0 = *a.e0;
        // the 1.01 covers the computed norms; float32 rounded upward throughout
        const float c = __fmul_ru(a.err_c, 1.01f);
        float U = 0.f;
        bool fin = true;
        for (int j = 0; j < a.k; ++j) {
            const int64_t o = static_cast<int64_t>(local) * a.KP + j;
            const float t = a.part_key[o];
            const int ix = a.part_idx[o];
            if (!(t < INFINITY) || ix < 0) {
                fin = false;
                break;
            }
            const float yn = a.ynorm[ix];
            U = fmaxf(U, __fadd_ru(__fadd_ru(xn, t), __fadd_ru(__fmul_ru(c, __fadd_ru(xn, yn)), e0)));
        }
        const float scale = 1.f + static_cast<float>(4 * a.d + 64) * 0x1p-24f;  // rounds up
        ub = fin ? __fsqrt_ru(__fmul_ru(U, __fadd_ru(scale, 0x1p-23f))) : INFINITY;
    }
    s_ub[tid] = ub;
    s_prow[tid] = row < a.row_end ? a.permX[row] : 0;
    // the second pass's shared threshold starts at the home list's KP-th key
    b_gthr[local] = row < a.row_end ? float_order(a.part_key[static_cast<int64_t>(local) * a.KP + a.KP - 1])
                                    : float_order(INFINITY);
    __syncthreads();

    // 2. The tile's hull per pivot (thread = pivot): the least d(x, p) - ub(x)
    //    and the largest d(x, p) + ub(x), d(x, p) widened by eps, in float32
    //    rounded outward (toward -inf for the least, +inf for the largest).
    {
        const float eps = static_cast<float>((a.d + 8) * 5.9604644775390625e-8);
        const float lo_f = __fsub_rd(1.f, eps), hi_f = __fadd_ru(1.f, eps);
        float A = INFINITY, Bv = -INFINITY;
        // the loads need no branch, so many are in flight: rows past the last
        // point (u < 0) read point 0's distances and do not use them
        const float *pd = a.pdX + tid;
#pragma unroll 16
        for (int r = 0; r < kBM; ++r) {
            const float u = s_ub[r];
            const float dx = pd[static_cast<int64_t>(s_prow[r]) * P];
            if (u >= 0.f) {
                A = fminf(A, __fsub_rd(__fmul_rd(dx, lo_f), u));
                Bv = fmaxf(Bv, __fadd_ru(__fmul_ru(dx, hi_f), u));
            }
        }
        s_A[tid] = A;
        s_B[tid] = Bv;
        // a pivot that separates no block from this hull is not worth testing
        // (an outlier tile's hull covers every block for most pivots)
        const bool useful = minH[tid] < A || maxL[tid] > Bv;
        const unsigned bal = __ballot_sync(0xffffffffu, useful);
        if (lane == 0) s_wc[warp] = __popc(bal);
        __syncthreads();
        int off = 0;
        for (int w = 0; w < warp; ++w) off += s_wc[w];
        if (useful) s_useful[off + __popc(bal & lanemask_lt())] = tid;
        const int nu = s_wc[0] + s_wc[1] + s_wc[2] + s_wc[3];
        __syncthreads();
        // pad to whole groups of 32 with repeats of the first useful pivot (a
        // repeated test changes nothing), so the tests below run 32 at a time
        const int npad = (nu + 31) / 32 * 32;
        if (tid >= nu && tid < npad) s_useful[tid] = s_useful[0];
        if (tid == 0) s_nuseful = npad;
    }
    __syncthreads();
    const int nuseful = s_nuseful;
    // the pivot nearest the whole tile (least B, the lower index on ties):
    // it separates most of the far blocks
    {
        unsigned long long kb = (static_cast<unsigned long long>(float_order(s_B[tid])) << 32) |
                                static_cast<unsigned>(tid);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) kb = min(kb, __shfl_xor_sync(0xffffffffu, kb, o));
        if (lane == 0) s_near[warp] = kb;
    }
    __syncthreads();
    const int pnear = static_cast<int>(min(min(s_near[0], s_near[1]), min(s_near[2], s_near[3])) & 0xffffffffu);
    // lane l tests pivot s_useful[32 g + l] of group g, whose (A, B) is
    // s_ABu[32 g + l]
    int pv[P / 32];
#pragma unroll
    for (int g = 0; g < P / 32; ++g) pv[g] = g * 32 + lane < nuseful ? s_useful[g * 32 + lane] : 0;
    if (tid < nuseful) s_ABu[tid] = make_float2(s_A[s_useful[tid]], s_B[s_useful[tid]]);

    // 3. Blocks outside the home range, outward from it (threads 0..63 to the
    //    right, 64..127 to the left, 64 offsets per step), kept unless one
    //    pivot separates them from every row.  The block's own pivot and the
    //    pivot nearest the tile are tried first (they separate most far
    //    blocks); the blocks they leave are then tested by a warp against
    //    all the useful pivots at once, a lane per pivot.
    const int h0 = home_lo[rt];
    const int right0 = h0 + nh, left0 = h0 - 1;
    int base = 0;
    for (int o0 = 0; right0 + o0 < a.col_tiles || left0 - o0 >= 0; o0 += 64) {
        const int o = o0 + (tid & 63);
        const int b = tid < 64 ? right0 + o : left0 - o;
        bool need = tid < 64 ? b < a.col_tiles : b >= 0;
        if (need) {
            const int p0 = bcell[b];
            need = !(Hm[static_cast<int64_t>(p0) * a.col_tiles + b] < s_A[p0] ||
                     Lm[static_cast<int64_t>(p0) * a.col_tiles + b] > s_B[p0]) &&
                   !(Hm[static_cast<int64_t>(pnear) * a.col_tiles + b] < s_A[pnear] ||
                     Lm[static_cast<int64_t>(pnear) * a.col_tiles + b] > s_B[pnear]);
        }
        // the blocks left, in thread order
        unsigned bal = __ballot_sync(0xffffffffu, need);
        if (lane == 0) s_wc[warp] = __popc(bal);
        __syncthreads();
        int ci = 0;
        for (int w = 0; w < warp; ++w) ci += s_wc[w];
        const int nc = s_wc[0] + s_wc[1] + s_wc[2] + s_wc[3];
        ci += __popc(bal & lanemask_lt());
        if (need) s_cand[ci] = b;
        __syncthreads();
        // every group's bounds of a block loaded at once (the loads, not the
        // tests, bound this loop)
        for (int c = warp; c < nc; c += kBM / 32) {
            const float2 *hl = HLt + static_cast<int64_t>(s_cand[c]) * P;
            float2 v[P / 32];
#pragma unroll
            for (int g = 0; g < P / 32; ++g)
                if (g * 32 < nuseful) v[g] = __ldg(hl + pv[g]);  // (H, L)
            bool sep = false;
#pragma unroll
            for (int g = 0; g < P / 32; ++g) {
                if (g * 32 < nuseful) {
                    const float2 ab = s_ABu[g * 32 + lane];
                    sep = sep || v[g].x < ab.x || v[g].y > ab.y;
                }
            }
            sep = __any_sync(0xffffffffu, sep);
            if (lane == 0) s_keep[c] = sep ? 0 : 1;
        }
        __syncthreads();
        if (need) need = s_keep[ci] != 0;
        bal = __ballot_sync(0xffffffffu, need);
        if (lane == 0) s_wc[warp] = __popc(bal);
        __syncthreads();
        int off = base;
        for (int w = 0; w < warp; ++w) off += s_wc[w];
        if (need) list[static_cast<int64_t>(rt) * a.col_tiles + off + __popc(bal & lanemask_lt())] = b;
        for (int w = 0; w < kBM / 32; ++w) base += s_wc[w];
        __syncthreads();
    }
    if (tid == 0) {
        count[rt] = base;
        slabs[rt] = 1 + (base + a.chunk_cap - 1) / a.chunk_cap;
        atomicAdd(a.blocks_total, static_cast<unsigned long long>(base + nh));
    }
}

// The row tiles by decreasing list length (ties: the lower tile first), so
// that a pruned pass, which dispatches its CTAs in this order, starts the
// longest first and ends on the shortest.  A thread per row tile counts the
// tiles that precede it in that order (the keys are distinct, so the counts
// are a permutation), reading all the lengths from shared memory.
constexpr int kOrderThreads = 128;
__global__ void __launch_bounds__(kOrderThreads) order_tiles_kernel(const int *__restrict__ count,
                                                                    int row_tiles,
                                                                    int *__restrict__ order) {
    __shared__ int4 s_cnt4[kOrderMax / 4];
    int *s_cnt = reinterpret_cast<int *>(s_cnt4);
    const int n4 = (row_tiles + 3) / 4;
    // past the last tile -1: lengths are never negative, so it precedes none
    for (int q = threadIdx.x; q < 4 * n4; q += kOrderThreads) s_cnt[q] = q < row_tiles ? count[q] : -1;
    __syncthreads();
    const int i = blockIdx.x * kOrderThreads + threadIdx.x;
    if (i >= row_tiles) return;
    const int ci = s_cnt[i];
    int rank = 0;
#pragma unroll 4
    for (int q = 0; q < n4; ++q) {
        const int4 c = s_cnt4[q];
        const int j = 4 * q;
        rank += (c.x > ci || (c.x == ci && j < i)) ? 1 : 0;
        rank += (c.y > ci || (c.y == ci && j + 1 < i)) ? 1 : 0;
        rank += (c.z > ci || (c.z == ci && j + 2 < i)) ? 1 : 0;
        rank += (c.w > ci || (c.w == ci && j + 3 < i)) ? 1 : 0;
    }
    order[rank] = i;
}

}  // namespace

cudaError_t launch_tile_order(const int *count, int row_tiles, int *order, cudaStream_t s) {
    if (row_tiles < 1 || row_tiles > kOrderMax) return cudaErrorInvalidValue;
    order_tiles_kernel<<<(row_tiles + kOrderThreads - 1) / kOrderThreads, kOrderThreads, 0, s>>>(
        count, row_tiles, order);
    return cudaGetLastError();
}

cudaError_t launch_prune_setup(const SpatialOrder &o, const PruneBufs &b, int m, int col_tiles,
                               int d, cudaStream_t s) {
    if (o.pivots != P) return cudaErrorInvalidValue;
    block_bounds_kernel<<<col_tiles, P, 0, s>>>(o.pdY, m, col_tiles, (d + 8.0) * 0x1p-24,
                                                o.cellY, o.permY, o.buckets, b.Lm, b.Hm,
                                                b.HLt, b.bcell);
    pivot_range_kernel<<<P, 256, 0, s>>>(b.Lm, b.Hm, col_tiles, b.minH, b.minH + P);
    count_extra_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_prune_home(const PruneHomeArgs &a, const PruneBufs &b, cudaStream_t s) {
    const SpatialOrder &o = *a.o;
    home_kernel<<<blocks_for(a.row_tiles, 128), 128, 0, s>>>(
        o.cellX, o.permX, o.startX, o.startY, a.n, a.col_tiles, a.row_tile0, a.row_tiles, a.nh,
        a.alias, b.home_lo, b.home);
    return cudaGetLastError();
}

cudaError_t launch_prune_lists(const PruneListArgs &a, const PruneBufs &b, cudaStream_t s) {
    prune_lists_kernel<<<a.row_tiles, kBM, 0, s>>>(a, b.Lm, b.Hm, b.HLt, b.bcell, b.home_lo,
                                                   b.list, b.count, b.slabs, b.gthr, b.minH,
                                                   b.minH + P);
    return cudaGetLastError();
}

}  // namespace hdbmst
