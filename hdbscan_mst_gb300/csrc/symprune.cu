// Pruning of the symmetric Boruvka scan (tc_sym.cu): which 128 x 128 block
// pairs of the set P can hold a pair that is some component's cheapest edge.
//
// Page "HDBSCAN" ("Exact shortcuts"): work is skipped only where a bound
// proves that it cannot change the result.  The bound here is the triangle
// inequality through pivots, as in the pruned k-NN (prune.cu): for a pivot p
// and points a, b, |d(a, p) - d(b, p)| <= d(a, b), so two blocks whose
// points' distances to p lie in [L_i, H_i] and [L_j, H_j] are at least
// LB(i, j) = max over p of max(L_j - H_i, L_i - H_j) apart.  A pair (a, b)
// of blocks i, j weighs at least its distance; if LB(i, j) exceeds the
// bounds theta of all components in both blocks, no pair of the two blocks
// is a cheapest edge of either end's component (theta only falls, and
// always weighs at least that component's cheapest edge).
//
// The bounds are tight only when the points of a block lie close together,
// so P is grouped by component and, within a component, in the spatial
// order of order.cu (nearest of 128 pivots, then distance bucket), and only
// once the component bounds are near their final values: a home pass first
// evaluates, for each row tile, the kSymHome blocks of other components with
// the least LB (which hold most components' cheapest edges), and the lists
// of the second pass are built from the bounds it leaves.
//
// Rounding.  Pivot distances are float32 direct differences within relative
// eps = (d + 8) 2^-24 of the true ones, and L, H are widened outward by eps;
// LB is formed with downward rounding.  The exact weight is at least its
// float32 distance, which is at least the true distance times (1 - (d + 4)
// 2^-24); a block pair is skipped only when LB (1 - 2^-16) exceeds the bound.
#include <cfloat>
#include <climits>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace hdbmst {

namespace {

constexpr int P = kPrunePivots;
constexpr int kRowsPerBlock = kBM;  // positions of a block

int blocks_for(int64_t n, int per) { return static_cast<int>(n > per ? (n + per - 1) / per : 1); }

// Compact index of every component label with points in P, and its first
// position.
__global__ void sym_compact_kernel(int n, const int *__restrict__ act_size,
                                   const int *__restrict__ act_start, int *__restrict__ kcount,
                                   int *__restrict__ cidx, int *__restrict__ cstart) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= n || act_size[c] == 0) return;
    const int k = atomicAdd(kcount, 1);
    if (k >= kSymMaxComps) return;  // the host checks the count first
    cidx[c] = k;
    cstart[k] = act_start[c];
}

// Per chunk of kSymChunk positions of the spatial order (one CTA; warp w
// takes the chunk's kSubChunk positions from w kSubChunk on), the points of
// each compact component that lie in P: lanes of one component add their
// number at once into the CTA's shared row, which is then written out whole
// (zeros included).
constexpr int kGroupWarps = 8, kSubChunk = kSymChunk / kGroupWarps;
static_assert(kSubChunk == 4 * 32, "four steps of 32 positions per warp");

// The compact component (or -1) and the point of the four steps of warp w.
__device__ __forceinline__ void sub_chunk_points(int p0, int p1, int warp, int lane,
                                                 const int *__restrict__ perm,
                                                 const unsigned char *__restrict__ act_flag,
                                                 const int *__restrict__ comp,
                                                 const int *__restrict__ cidx, int (&x)[4],
                                                 int (&k)[4]) {
    const int s0 = p0 + warp * kSubChunk + lane;
#pragma unroll
    for (int u = 0; u < 4; ++u) x[u] = s0 + 32 * u < p1 ? perm[s0 + 32 * u] : -1;
#pragma unroll
    for (int u = 0; u < 4; ++u) k[u] = (x[u] >= 0 && act_flag[x[u]]) ? comp[x[u]] : -1;
#pragma unroll
    for (int u = 0; u < 4; ++u) k[u] = k[u] >= 0 ? cidx[k[u]] : -1;
}

__global__ void __launch_bounds__(kGroupWarps * 32)
    sym_chunk_count_kernel(int n, const int *__restrict__ perm,
                           const unsigned char *__restrict__ act_flag,
                           const int *__restrict__ comp, const int *__restrict__ cidx,
                           int *__restrict__ off) {
    __shared__ int s_cnt[kSymMaxComps];
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int chunk = blockIdx.x;
    const int p0 = chunk * kSymChunk, p1 = min(p0 + kSymChunk, n);
    for (int k = t; k < kSymMaxComps; k += kGroupWarps * 32) s_cnt[k] = 0;
    __syncthreads();
    int x[4], k[4];
    sub_chunk_points(p0, p1, warp, lane, perm, act_flag, comp, cidx, x, k);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const unsigned peers = __match_any_sync(0xffffffffu, k[u]);
        if (k[u] >= 0 && lane == __ffs(peers) - 1) atomicAdd(&s_cnt[k[u]], __popc(peers));
    }
    __syncthreads();
    int *row = off + static_cast<int64_t>(chunk) * kSymMaxComps;
    for (int c = t; c < kSymMaxComps; c += kGroupWarps * 32) row[c] = s_cnt[c];
}

// Per compact component, the running position at the start of each chunk.
__global__ void sym_chunk_scan_kernel(int chunks, int ncomp, const int *__restrict__ cstart,
                                      int *__restrict__ off) {
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= ncomp) return;
    int run = cstart[k];
    for (int ch = 0; ch < chunks; ++ch) {
        int *e = off + static_cast<int64_t>(ch) * kSymMaxComps + k;
        const int cnt = *e;
        *e = run;
        run += cnt;
    }
}

// Positions in chunk order and, within a chunk, in spatial order (one CTA
// per chunk): each warp counts its sub-chunk's points per component, a
// prefix over the warps per component gives each warp's first positions from
// the chunk's, and each warp then places its points 32 at a time, lanes of
// one component at consecutive positions in lane order.
__global__ void __launch_bounds__(kGroupWarps * 32)
    sym_scatter_kernel(int n, const int *__restrict__ perm,
                       const unsigned char *__restrict__ act_flag,
                       const int *__restrict__ comp, const int *__restrict__ cidx,
                       const int *__restrict__ off, int *__restrict__ act_idx) {
    __shared__ int s_pos[kGroupWarps][kSymMaxComps];
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int chunk = blockIdx.x;
    const int p0 = chunk * kSymChunk, p1 = min(p0 + kSymChunk, n);
    for (int c = t; c < kGroupWarps * kSymMaxComps; c += kGroupWarps * 32) (&s_pos[0][0])[c] = 0;
    __syncthreads();
    int x[4], k[4];
    sub_chunk_points(p0, p1, warp, lane, perm, act_flag, comp, cidx, x, k);
    int *own = s_pos[warp];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const unsigned peers = __match_any_sync(0xffffffffu, k[u]);
        if (k[u] >= 0 && lane == __ffs(peers) - 1) own[k[u]] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    const int *row = off + static_cast<int64_t>(chunk) * kSymMaxComps;
    for (int c = t; c < kSymMaxComps; c += kGroupWarps * 32) {
        int run = row[c];
#pragma unroll
        for (int w = 0; w < kGroupWarps; ++w) {
            const int cnt = s_pos[w][c];
            s_pos[w][c] = run;
            run += cnt;
        }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const unsigned peers = __match_any_sync(0xffffffffu, k[u]);
        const int base = k[u] >= 0 ? own[k[u]] : 0;
        __syncwarp();
        if (k[u] >= 0) {
            act_idx[base + __popc(peers & lanemask_lt())] = x[u];
            if (lane == __ffs(peers) - 1) own[k[u]] = base + __popc(peers);
        }
        __syncwarp();
    }
}

// Per block b of P (one CTA, thread = pivot): the least and largest pivot
// distance of its points, widened outward by eps; and bcomp[b], the
// component of a block whose points all have the same one (else -1).
__global__ void __launch_bounds__(P) sym_bounds_kernel(int np, const int *__restrict__ act_idx,
                                                       const int *__restrict__ pcomp,
                                                       const float *__restrict__ pd, double eps,
                                                       float *__restrict__ Lb,
                                                       float *__restrict__ Hb,
                                                       int *__restrict__ bcomp) {
    static_assert(kRowsPerBlock == P, "one position per thread");
    __shared__ int s_pt[kRowsPerBlock];
    const int b = blockIdx.x, p = threadIdx.x;
    const int q0 = b * kRowsPerBlock, q1 = min(q0 + kRowsPerBlock, np);
    // the block's points, and whether they all share the first one's component
    const bool in = q0 + p < q1;
    s_pt[p] = in ? act_idx[q0 + p] : 0;
    const int c0 = pcomp[q0];
    const bool same = __syncthreads_and(!in || pcomp[q0 + p] == c0);
    float lo = INFINITY, hi = -INFINITY;
#pragma unroll 8
    for (int q = 0; q < q1 - q0; ++q) {
        const float v = pd[static_cast<int64_t>(s_pt[q]) * P + p];
        lo = fminf(lo, v);
        hi = fmaxf(hi, v);
    }
    Lb[static_cast<int64_t>(b) * P + p] = __double2float_rd(static_cast<double>(lo) * (1.0 - eps));
    Hb[static_cast<int64_t>(b) * P + p] = __double2float_ru(static_cast<double>(hi) * (1.0 + eps));
    if (p == 0) bcomp[b] = same ? c0 : -1;
}

// LB[i][j] for all block pairs (LB is symmetric: only tiles with j0 >= i0
// are computed, and written to both halves).  A CTA of 256 threads takes 64
// x 64 pairs, each thread 4 x 4, with the pivots staged 32 at a time (rows
// padded by one word: the staging writes a pivot per lane, which would
// otherwise all fall on one bank).
constexpr int kLbTile = 64, kLbPiv = 32, kLbPad = kLbTile + 1;
__global__ void __launch_bounds__(256) sym_lb_kernel(int blocks, const float *__restrict__ Lb,
                                                     const float *__restrict__ Hb,
                                                     float *__restrict__ LB) {
    const int ti = blockIdx.y, tj = blockIdx.x;
    if (tj < ti) return;
    __shared__ float sLi[kLbPiv][kLbPad], sHi[kLbPiv][kLbPad], sLj[kLbPiv][kLbPad],
        sHj[kLbPiv][kLbPad];
    const int i0 = ti * kLbTile, j0 = tj * kLbTile;
    const int t = threadIdx.x, ty = t >> 4, tx = t & 15;
    float lb[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) lb[a][c] = 0.f;
    for (int p0 = 0; p0 < P; p0 += kLbPiv) {
        __syncthreads();
        for (int e = t; e < kLbTile * kLbPiv; e += 256) {
            const int r = e / kLbPiv, q = e % kLbPiv;
            const int bi = min(i0 + r, blocks - 1), bj = min(j0 + r, blocks - 1);
            sLi[q][r] = Lb[static_cast<int64_t>(bi) * P + p0 + q];
            sHi[q][r] = Hb[static_cast<int64_t>(bi) * P + p0 + q];
            sLj[q][r] = Lb[static_cast<int64_t>(bj) * P + p0 + q];
            sHj[q][r] = Hb[static_cast<int64_t>(bj) * P + p0 + q];
        }
        __syncthreads();
#pragma unroll 4
        for (int q = 0; q < kLbPiv; ++q) {
            float li[4], hi[4], lj[4], hj[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                li[a] = sLi[q][ty + 16 * a];
                hi[a] = sHi[q][ty + 16 * a];
                lj[a] = sLj[q][tx + 16 * a];
                hj[a] = sHj[q][tx + 16 * a];
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    lb[a][c] = fmaxf(lb[a][c], fmaxf(__fsub_rd(lj[c], hi[a]), __fsub_rd(li[a], hj[c])));
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int i = i0 + ty + 16 * a, j = j0 + tx + 16 * c;
            if (i < blocks && j < blocks) {
                LB[static_cast<int64_t>(i) * blocks + j] = lb[a][c];
                LB[static_cast<int64_t>(j) * blocks + i] = lb[a][c];
            }
        }
}

__device__ __forceinline__ bool own_pair(const int *bcomp, int i, int j) {
    const int ci = bcomp[i];
    return ci >= 0 && bcomp[j] == ci;
}

// Home list of row tile i (one CTA): its kSymHome blocks of least LB that
// are not wholly inside its own component (block i itself included when it
// holds two components).  Each thread keeps its best kSymHome keys (LB bits,
// block); the CTA then pops the least head kSymHome times.
constexpr int kHomeThreads = 256;
__global__ void __launch_bounds__(kHomeThreads) sym_home_kernel(int blocks,
                                                                const float *__restrict__ LB,
                                                                const int *__restrict__ bcomp,
                                                                int *__restrict__ home,
                                                                int *__restrict__ hcount,
                                                                int *__restrict__ hkey) {
    __shared__ unsigned long long s_min[kHomeThreads / 32];
    __shared__ unsigned long long s_win;
    const int i = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    unsigned long long best[kSymHome];
#pragma unroll
    for (int q = 0; q < kSymHome; ++q) best[q] = kNoKey;
    for (int j = t; j < blocks; j += kHomeThreads) {
        if (own_pair(bcomp, i, j)) continue;
        const unsigned long long key =
            (static_cast<unsigned long long>(__float_as_uint(LB[static_cast<int64_t>(i) * blocks + j])) << 32) |
            static_cast<unsigned>(j);
        if (key < best[kSymHome - 1]) {
            best[kSymHome - 1] = key;
#pragma unroll
            for (int q = kSymHome - 1; q > 0; --q) {
                const unsigned long long lo = min(best[q - 1], best[q]), hi = max(best[q - 1], best[q]);
                best[q - 1] = lo;
                best[q] = hi;
            }
        }
    }
    int head = 0, cnt = 0;
    for (int r = 0; r < kSymHome; ++r) {
        unsigned long long h = head < kSymHome ? best[0] : kNoKey;
#pragma unroll
        for (int q = 1; q < kSymHome; ++q)
            if (q == head) h = best[q];
        unsigned long long m = h;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = min(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) s_min[warp] = m;
        __syncthreads();
        if (t == 0) {
            unsigned long long w = s_min[0];
            for (int q = 1; q < kHomeThreads / 32; ++q) w = min(w, s_min[q]);
            s_win = w;
        }
        __syncthreads();
        const unsigned long long w = s_win;
        if (w == kNoKey) break;
        if (h == w) ++head;  // keys are distinct (block index)
        if (t == 0) home[static_cast<int64_t>(i) * kSymHome + cnt] = static_cast<int>(w & 0xffffffffu);
        // the home pass's work estimate: the nearer the tile's nearest block
        // of another component, the more pairs it records (a bound's bits,
        // non-negative, order like the bound)
        if (t == 0 && cnt == 0) hkey[i] = 0x7fffffff - static_cast<int>(min(static_cast<unsigned>(w >> 32), 0x7fffffffu));
        ++cnt;
        __syncthreads();
    }
    if (t == 0) {
        hcount[i] = cnt;
        if (cnt == 0) hkey[i] = 0;
    }
}

// bth[b]: the largest live bound over the components of block b's points.
__global__ void __launch_bounds__(kRowsPerBlock) sym_block_theta_kernel(int np,
                                                                        const int *__restrict__ pcomp,
                                                                        const unsigned *__restrict__ theta,
                                                                        float *__restrict__ bth) {
    __shared__ unsigned s_max[kRowsPerBlock / 32];
    const int b = blockIdx.x, t = threadIdx.x;
    const int q = b * kRowsPerBlock + t;
    unsigned m = q < np ? __ldcg(theta + pcomp[q]) : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((t & 31) == 0) s_max[t >> 5] = m;
    __syncthreads();
    if (t == 0) {
        unsigned w = s_max[0];
        for (int k = 1; k < kRowsPerBlock / 32; ++k) w = max(w, s_max[k]);
        bth[b] = __uint_as_float(w);
    }
}

// List of row tile i (one CTA, order kept): the blocks j >= i, not wholly
// inside i's component and not in its home list, whose bound LB (1 - 2^-16)
// does not exceed max(bth[i], bth[j]).
constexpr int kListThreads = 256;
__global__ void __launch_bounds__(kListThreads) sym_list_kernel(int blocks,
                                                                const float *__restrict__ LB,
                                                                const float *__restrict__ bth,
                                                                const int *__restrict__ bcomp,
                                                                const int *__restrict__ home,
                                                                const int *__restrict__ hcount,
                                                                int *__restrict__ list,
                                                                int *__restrict__ lcount) {
    __shared__ int s_home[kSymHome];
    __shared__ int s_warp[kListThreads / 32];
    const int i = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int hc = hcount[i];
    if (t < kSymHome) s_home[t] = t < hc ? home[static_cast<int64_t>(i) * kSymHome + t] : -1;
    __syncthreads();
    const float thi = bth[i];
    int cnt = 0;
    for (int j0 = i; j0 < blocks; j0 += kListThreads) {
        const int j = j0 + t;
        bool keep = false;
        if (j < blocks && !own_pair(bcomp, i, j)) {
            const float lb = __fmul_rd(LB[static_cast<int64_t>(i) * blocks + j], 1.f - 0x1p-16f);
            keep = !(lb > fmaxf(thi, bth[j]));
#pragma unroll
            for (int q = 0; q < kSymHome; ++q) keep = keep && s_home[q] != j;
        }
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        if (lane == 0) s_warp[warp] = __popc(bal);
        __syncthreads();
        int before = 0, total = 0;
        for (int w = 0; w < kListThreads / 32; ++w) {
            before += w < warp ? s_warp[w] : 0;
            total += s_warp[w];
        }
        if (keep) list[static_cast<int64_t>(i) * blocks + cnt + before + __popc(bal & lanemask_lt())] = j;
        cnt += total;
        __syncthreads();
    }
    if (t == 0) lcount[i] = cnt;
}

}  // namespace

cudaError_t launch_sym_group(const SymPruneBufs &b, int n, const unsigned char *act_flag,
                             const int *comp, const int *act_start, const int *act_size,
                             int *act_idx, cudaStream_t s) {
    const int chunks = blocks_for(n, kSymChunk);
    cudaError_t e = cudaMemsetAsync(b.kcount, 0, sizeof(int), s);
    if (e != cudaSuccess) return e;
    sym_compact_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, act_size, act_start, b.kcount, b.cidx,
                                                          b.cstart);
    sym_chunk_count_kernel<<<chunks, kGroupWarps * 32, 0, s>>>(n, b.order.permY, act_flag, comp,
                                                              b.cidx, b.off);
    sym_chunk_scan_kernel<<<blocks_for(kSymMaxComps, 256), 256, 0, s>>>(chunks, kSymMaxComps,
                                                                        b.cstart, b.off);
    sym_scatter_kernel<<<chunks, kGroupWarps * 32, 0, s>>>(n, b.order.permY, act_flag, comp,
                                                          b.cidx, b.off, act_idx);
    count_extra_launches(3);
    return cudaGetLastError();
}

cudaError_t launch_sym_blocks(const SymPruneBufs &b, int np, int blocks, const int *act_idx,
                              const int *pcomp, int d, cudaStream_t s) {
    const double eps = (d + 8.0) * 0x1p-24;
    sym_bounds_kernel<<<blocks, P, 0, s>>>(np, act_idx, pcomp, b.order.pdY, eps, b.Lb, b.Hb,
                                           b.bcomp);
    const int g = (blocks + kLbTile - 1) / kLbTile;
    sym_lb_kernel<<<dim3(g, g), 256, 0, s>>>(blocks, b.Lb, b.Hb, b.LB);
    sym_home_kernel<<<blocks, kHomeThreads, 0, s>>>(blocks, b.LB, b.bcomp, b.home, b.hcount,
                                                     b.hkey);
    count_extra_launches(2);
    return cudaGetLastError();
}

cudaError_t launch_sym_lists(const SymPruneBufs &b, int np, int blocks, const int *pcomp,
                             const unsigned *theta, int d, cudaStream_t s) {
    (void)d;
    sym_block_theta_kernel<<<blocks, kRowsPerBlock, 0, s>>>(np, pcomp, theta, b.bth);
    sym_list_kernel<<<blocks, kListThreads, 0, s>>>(blocks, b.LB, b.bth, b.bcomp, b.home,
                                                    b.hcount, b.list, b.lcount);
    count_extra_launches(1);
    return cudaGetLastError();
}

}  // namespace hdbmst
