// K1 / K1r / K1x: exact k-nearest neighbours.
//
// Page "Kilosort4 clustering and matching" (neuro-kitchen dsp-kitchen
// gpu/clustering), section "k-nearest neighbours are a matrix product": with
// |x - y|^2 = |x|^2 + |y|^2 - 2 x.y the distances of a block of rows to a set
// are one matrix product plus two norm vectors, a small selection keeps the
// smallest per row, and rows go in chunks so scratch stays bounded.  Page
// "HDBSCAN" (gpu/hdbscan), section "The hang": the nearest list is kept by a
// fixed sequence of compare-and-swaps, no loop waits on a flag, and equal
// distances keep their order (lowest index first).
//
// The GB300 design:
//  * K1 (knn_tile_kernel): a 128 x 128 register-blocked FFMA tile (8 x 8 per
//    thread) over feature chunks of 16 staged in shared memory by cp.async
//    double buffering.  The product never reaches global memory: per pair the
//    epilogue forms t = |y|^2 - 2 x.y (the row's |x|^2 is a constant shift)
//    and tests it against the row's current KP-th best.  A warp owns 16 whole
//    rows, so candidates go to warp-private shared buffers and one lane per
//    row folds them into the row's sorted list with unrolled compare-and-swap;
//    no block-wide barrier is spent on selection.  Columns are split across
//    CTAs so the grid fills every SM; each CTA writes a partial list.
//  * K1r (knn_refine_kernel): merges the partial lists, re-evaluates every kept
//    candidate with the library's exact distance (direct differences), sorts
//    by (dist, index) and proves, from a bound on the expansion's rounding
//    error, that no dropped column could enter the top k.  Rows it cannot prove
//    are queued for K1x.
//  * K1x (knn_exact_kernel): searches queued rows again with the exact
//    distance over every column.
#include <cfloat>
#include <climits>
#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "tile.cuh"

namespace hdbmst {

namespace {

constexpr int kCap = 16;               // candidate slots per row per merge
constexpr int kMaxPass = kBN / kCap + 2;  // pushes per tile are bounded by kBN per row

template <int KP>
struct TileSmem {
    TileBuffers T;
    float lkey[kBM][KP + 1];  // +1: rows of consecutive lanes fall in different banks
    int lidx[kBM][KP + 1];
    float ckey[kBM][kCap + 1];
    int cidx[kBM][kCap + 1];
    int ccnt[kBM];
    float tau[kBM];
};

// The 16 local rows that warp w owns (thread rows ty = 2w and 2w + 1).
__device__ __forceinline__ int warp_row(int w, int q) { return (q < 8 ? 0 : 56) + w * 8 + q; }

__device__ __forceinline__ bool key_less(float a, int ai, float b, int bi) {
    return a < b || (a == b && ai < bi);
}

// Fold row r's queued candidates into its sorted list.  Each insertion is
// the same fixed compare-and-swap pass as a register list would take (the
// newcomer replaces the last entry and sinks), done on the row's shared
// memory slots so the 64 tile accumulators keep their registers.  The pass
// stops early once the newcomer is in place; its length is bounded by KP.
template <int KP>
__device__ __forceinline__ void merge_row(TileSmem<KP> &S, int r) {
    int cnt = S.ccnt[r];
    if (cnt == 0) return;
    cnt = min(cnt, kCap);
    S.ccnt[r] = 0;
    float *lk = S.lkey[r];
    int *li = S.lidx[r];
    for (int c = 0; c < cnt; ++c) {
        const float t = S.ckey[r][c];
        const int j = S.cidx[r][c];
        if (!key_less(t, j, lk[KP - 1], li[KP - 1])) continue;
        int p = KP - 1;
#pragma unroll 4
        for (int s = 0; s < KP - 1; ++s) {
            const float pk = lk[p - 1];
            const int pi = li[p - 1];
            if (!key_less(t, j, pk, pi)) break;
            lk[p] = pk;
            li[p] = pi;
            --p;
        }
        lk[p] = t;
        li[p] = j;
    }
    S.tau[r] = lk[KP - 1];
}

// Rare path of the selection: some row's buffer filled up (in practice only in
// a CTA's first tiles, while the thresholds are still loose).  Retry the
// pending pairs against the tightened thresholds.  Each pass stores kCap
// candidates of every row that still has pending ones, so kMaxPass passes
// always suffice; the bound is a constant, never a flag.  Kept out of line:
// it takes the tile's values through a local copy so that the main loop's
// accumulators never leave registers.
template <int KP>
__device__ __noinline__ void overflow_retry(TileSmem<KP> &S, const float *tv,
                                            unsigned long long pend, int col0, int warp,
                                            int lane, int ty, int tx) {
    for (int pass = 1; pass < kMaxPass; ++pass) {
        if (!__any_sync(0xffffffffu, pend != 0ull)) break;
        unsigned long long rem = pend;
        for (int it = 0; it < 64 && rem != 0ull; ++it) {
            const int b = __ffsll(static_cast<long long>(rem)) - 1;
            rem &= rem - 1ull;
            const int i = b >> 3, j = b & 7;
            const int r = row_of(ty, i);
            const float t = tv[b];
            if (t < S.tau[r]) {
                const int pos = atomicAdd(&S.ccnt[r], 1);
                if (pos < kCap) {
                    S.ckey[r][pos] = t;
                    S.cidx[r][pos] = col0 + col_of(tx, j);
                    pend &= ~(1ull << b);
                }
            } else {
                pend &= ~(1ull << b);
            }
        }
        __syncwarp();
        if (lane < 16) merge_row<KP>(S, warp_row(warp, lane));
        __syncwarp();
    }
}

// Selection epilogue of one 128-column tile, run by each warp on its own rows.
template <int KP>
__device__ __forceinline__ void tile_epilogue(TileSmem<KP> &S, float (&acc)[8][8],
                                              const float *__restrict__ ynorm, int col0,
                                              int warp, int lane, int ty, int tx) {
    float yn[8];
    {
        const float4 v0 = __ldg(reinterpret_cast<const float4 *>(ynorm + col0 + tx * 4));
        const float4 v1 = __ldg(reinterpret_cast<const float4 *>(ynorm + col0 + 64 + tx * 4));
        yn[0] = v0.x; yn[1] = v0.y; yn[2] = v0.z; yn[3] = v0.w;
        yn[4] = v1.x; yn[5] = v1.y; yn[6] = v1.z; yn[7] = v1.w;
    }
    unsigned long long pend = 0ull;  // pairs that found their row's buffer full
    bool pushed = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = row_of(ty, i);
        const float tau = S.tau[r];
        float mn = INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            acc[i][j] = __fmaf_rn(-2.f, acc[i][j], yn[j]);
            mn = fminf(mn, acc[i][j]);
        }
        if (mn < tau) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (acc[i][j] < tau) {
                    const int pos = atomicAdd(&S.ccnt[r], 1);
                    if (pos < kCap) {
                        S.ckey[r][pos] = acc[i][j];
                        S.cidx[r][pos] = col0 + col_of(tx, j);
                        pushed = true;
                    } else {
                        pend |= 1ull << (i * 8 + j);
                    }
                }
            }
        }
    }
    if (!__any_sync(0xffffffffu, pushed || pend != 0ull)) return;
    __syncwarp();
    if (lane < 16) merge_row<KP>(S, warp_row(warp, lane));
    __syncwarp();
    if (__any_sync(0xffffffffu, pend != 0ull)) {
        float tv[64];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) tv[i * 8 + j] = acc[i][j];
        overflow_retry<KP>(S, tv, pend, col0, warp, lane, ty, tx);
    }
}

template <int KP>
__global__ void __launch_bounds__(kThreads, 2) knn_tile_kernel(const KnnTileArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    TileSmem<KP> &S = *reinterpret_cast<TileSmem<KP> *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ty = tid >> 4, tx = tid & 15;
    const int row_tile = blockIdx.x;
    const int split = blockIdx.y;
    const int r0 = a.row_base + row_tile * kBM;
    const int ct_begin = split * a.tiles_per_split;
    const int ct_end = min(ct_begin + a.tiles_per_split, a.col_tiles);

    if (lane < 16) {
        const int r = warp_row(warp, lane);
#pragma unroll
        for (int p = 0; p < KP; ++p) {
            S.lkey[r][p] = INFINITY;
            S.lidx[r][p] = INT_MAX;
        }
        S.ccnt[r] = 0;
        S.tau[r] = INFINITY;
    }
    __syncwarp();

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    tile_pipeline(S.T, a.Xf, a.ldx, r0, a.Yf, a.ldy, ct_begin, ct_end, 0, 0, a.dk, acc,
                  [&](float (&ac)[8][8], int ct) {
        tile_epilogue<KP>(S, ac, a.ynorm, ct * kBN, warp, lane, ty, tx);
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) ac[i][j] = 0.f;
    });
    __syncwarp();
    if (lane < 16) {
        const int r = warp_row(warp, lane);
        const int local = row_tile * kBM + r;
        if (a.row_base + local < a.row_end) {
            const int64_t o = (static_cast<int64_t>(split) * a.chunk_rows_pad + local) * KP;
#pragma unroll
            for (int p = 0; p < KP; ++p) {
                a.part_key[o + p] = S.lkey[r][p];
                a.part_idx[o + p] = S.lidx[r][p];
            }
        }
    }
}

// ------------------------------------------------------------------ refine

// Groups of KP lanes; each group owns one query row.  The candidates' rows
// are read kSegF features at a time into shared memory (rows padded to
// kSegStride floats: the lanes' 16-byte reads of their own rows then fall on
// distinct banks in each quarter warp); the query row (up to kRefineXMax
// features) is copied whole at the start.
constexpr int kSegF = 32, kSegStride = 36, kRefineXMax = 192;

template <int KP>
__global__ void __launch_bounds__(128) knn_refine_kernel(const KnnRefineArgs a) {
    __shared__ float sel_t[128];
    __shared__ int sel_j[128];
    __shared__ __align__(16) float s_seg[2][128 / KP][KP][kSegStride];
    __shared__ __align__(16) float s_x[128 / KP][kRefineXMax];
    const int gl = threadIdx.x % KP;
    const int group = threadIdx.x / KP;
    const int local = blockIdx.x * (128 / KP) + group;
    const int row = a.row_base + local;
    const bool active = row < a.row_end;
    const int leader = (threadIdx.x & 31) & ~(KP - 1);
    // the query row, in flight while the lists merge
    const bool x_smem = a.dk <= kRefineXMax;
    if (x_smem && active)
        for (int q = gl; q < a.dk / 4; q += KP)
            cp_async16(&s_x[group][q * 4], a.Xp + static_cast<int64_t>(row) * a.dk + q * 4);
    cp_async_commit();

    // 1. Merge the sorted partial lists of the splits into the KP best by
    //    (t, index), the KP lanes of the row together: lane p holds entry p
    //    of the running list; a further list is merged by pairing entry p
    //    with the other's entry KP - 1 - p (the KP lesser of the pairs are
    //    the KP least of both, as a bitonic sequence) and a half-cleaner
    //    cascade over the lanes.  Keys are (t, index) as order-preserving
    //    bits (t + 0 turns -0 into +0, which key_less treats alike).
    float A = INFINITY;
    const int slabs = (a.tile_slabs && active) ? min(a.splits, a.tile_slabs[local / kBM]) : a.splits;
    const auto load_key = [&](int s, int pos) -> unsigned long long {
        const int64_t o = (static_cast<int64_t>(s) * a.chunk_rows_pad + local) * KP + pos;
        const float t = __fadd_rn(a.part_key[o], 0.f);
        return (static_cast<unsigned long long>(float_order(t)) << 32) |
               static_cast<unsigned>(a.part_idx[o]);
    };
    constexpr unsigned long long kEmpty = 0xFF8000007FFFFFFFull;  // (+inf, INT_MAX)
    unsigned long long mk = active ? load_key(0, gl) : kEmpty;
    // every lane of the warp runs the same merges (the shuffles); the
    // further lists are loaded four at a time
    const int slabs_w = __reduce_max_sync(0xffffffffu, active ? slabs : 0);
    for (int s0 = 1; s0 < slabs_w; s0 += 4) {
        unsigned long long o[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            o[u] = (active && s0 + u < slabs) ? load_key(s0 + u, KP - 1 - gl) : kEmpty;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (s0 + u >= slabs_w) break;
            mk = min(mk, o[u]);
#pragma unroll
            for (int h = KP / 2; h > 0; h >>= 1) {
                const unsigned long long q = __shfl_xor_sync(0xffffffffu, mk, h);
                mk = (gl & h) ? max(mk, q) : min(mk, q);
            }
        }
    }
    sel_t[group * KP + gl] = order_float(static_cast<unsigned>(mk >> 32));
    sel_j[group * KP + gl] = static_cast<int>(mk & 0xffffffffu);
    if (gl == KP - 1) A = sel_t[group * KP + KP - 1];
    __syncwarp();
    A = __shfl_sync(0xffffffffu, A, leader + KP - 1);

    // 2. Exact distance of every kept candidate that can still reach the top
    //    k.  The first k by t each have a true squared distance of at most
    //    xn + t + c (xn + yn) + e0; a candidate whose lower bound xn + t -
    //    c (xn + yn) - e0 exceeds the largest of those by more than the float32
    //    evaluation of dist() can move (both sides, rounded outward) ranks
    //    after the k-th and needs no exact distance (its key stays last).
    const int j = sel_j[group * KP + gl];
    bool need = active && j >= 0 && j < a.m;
    {
        const float xn = active ? a.xnorm[row] : 0.f;
        const float tj = sel_t[group * KP + gl];
        float hi = -INFINITY, lo = INFINITY;
        if (need) {
            const float err = __fadd_ru(__fmul_ru(a.err_c, __fadd_ru(xn, a.ynorm[j])), *a.e0);
            if (gl < a.k) hi = __fadd_ru(tj, err);
            lo = __fsub_rd(tj, err);
        }
#pragma unroll
        for (int o = 1; o < KP; o <<= 1) hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        const float mg = static_cast<float>(a.d + 8) * 0x1p-24f;
        if (need && gl >= a.k &&
            __fmul_rd(__fadd_rd(lo, xn), __fsub_rd(1.f, mg)) > __fmul_ru(__fadd_ru(hi, xn), __fadd_ru(1.f, mg)))
            need = false;
    }
    //    The group copies its candidates' rows kSegF features at a time,
    //    eight lanes per candidate segment (whole 32-byte sectors), two
    //    stages in flight; each lane then runs its own candidate's chain in
    //    feature order from shared memory.
    unsigned long long key = kNoKey;
    {
        const unsigned needs = __ballot_sync(0xffffffffu, need) >> leader;  // bit p: candidate p
        const float4 *xp = reinterpret_cast<const float4 *>(a.Xp + static_cast<int64_t>(active ? row : 0) * a.dk);
        const int nseg = (a.dk + kSegF - 1) / kSegF;
        const auto issue = [&](int c) {
            const int f0 = c * kSegF, w = min(kSegF, a.dk - f0), q = gl & 7;
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int p = it * (KP / 8) + (gl >> 3);
                if (((needs >> p) & 1u) && q * 4 < w)
                    cp_async16_ca(&s_seg[c & 1][group][p][q * 4],
                                  a.Yp + static_cast<int64_t>(sel_j[group * KP + p]) * a.dk + f0 + q * 4);
            }
            cp_async_commit();
        };
        float acc = 0.f;
        issue(0);
        for (int c = 0; c < nseg; ++c) {
            if (c + 1 < nseg) {
                issue(c + 1);
                cp_async_wait_one();
            } else {
                cp_async_wait_all();
            }
            __syncwarp();
            if (need) {
                const int f0 = c * kSegF, w = min(kSegF, a.dk - f0);
                const float *ys = &s_seg[c & 1][group][gl][0];
#pragma unroll 4
                for (int f = 0; f < w; f += 4) {
                    const float4 x = x_smem ? *reinterpret_cast<const float4 *>(&s_x[group][f0 + f])
                                            : __ldg(xp + (f0 + f) / 4);
                    const float4 y = *reinterpret_cast<const float4 *>(ys + f);
                    acc = sqdiff_fma(x.x, y.x, acc);
                    acc = sqdiff_fma(x.y, y.y, acc);
                    acc = sqdiff_fma(x.z, y.z, acc);
                    acc = sqdiff_fma(x.w, y.w, acc);
                }
            }
            __syncwarp();  // every lane is done with the stage before it is refilled
        }
        // rank by the caller's column index (the packed order may be spatial)
        if (need) key = key64(__fsqrt_rn(acc), static_cast<unsigned>(a.permY ? a.permY[j] : j));
    }

    // 3. Bitonic sort of the group's KP keys, ascending.
#pragma unroll
    for (int size = 2; size <= KP; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, stride);
            const bool up = (gl & size) == 0;
            const bool lower = (gl & stride) == 0;
            key = (lower == up) ? min(key, other) : max(key, other);
        }
    }

    if (!active) return;
    const int orow = a.permX ? a.permX[row] : row;  // the caller's row
    const int64_t o = static_cast<int64_t>(orow) * a.k;
    if (gl < a.k) {
        a.out_idx[o + gl] = static_cast<int32_t>(key_i(key));
        a.out_dist[o + gl] = key_w(key);
    }
    if (a.out_core && gl == a.core_rank - 1) a.out_core[orow] = key_w(key);

    // 4. Proof that the kept set holds the exact top k.  Every dropped column
    //    z has computed t_z >= A (A = the KP-th kept t).  The ranking error of
    //    t is at most err_coef (|x|^2 + |z|^2), so z's true squared distance is
    //    at least |x|^2 + A - err_coef (|x|^2 + |z|^2); by Cauchy-Schwarz it is
    //    also at least (|z| - |x|)^2.  With T = dist_k^2 M (M covers the exact
    //    float32 evaluation, (1 - (d + 3) u), and strict sqrt ordering,
    //    16 u), every z with |z|^2 >= nb_c = (|x| + sqrt(T))^2 is beyond T by
    //    the second bound, and every other z by the first as soon as
    //    |x|^2 + A - err_coef (|x|^2 + nb_c) > T.  Then no dropped column can
    //    rank in the top k.  The bound needs no maximum over all columns.  The
    //    FP16 operands add an absolute part e0 to the ranking error.  Every
    //    step is float32 rounded in the safe direction (proof_* in common.cuh).
    if (gl == a.k - 1 && A < INFINITY) {
        const float T = proof_T_up(key_w(key), a.d);
        if (!(proof_lhs_down(A, a.xnorm[row], T, a.err_c, *a.e0) > T)) {
            const int pos = atomicAdd(a.fb_count, 1);
            a.fb_rows[pos] = row;
        }
    }
}

// ------------------------------------------------------------------ exact rows

template <int KP>
__global__ void __launch_bounds__(256) knn_exact_kernel(const KnnExactArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned long long *lists = reinterpret_cast<unsigned long long *>(smem_raw);  // [256][KP]
    float *xrow = reinterpret_cast<float *>(lists + 256 * KP);                       // [dk]
    __shared__ unsigned long long wmin[8];
    const int tid = threadIdx.x;
    const int count = *a.fb_count;
    for (int f = a.rows_cap + blockIdx.x; f < count; f += gridDim.x) {
        const int row = a.fb_rows[f];
        for (int q = tid; q < a.dk; q += 256) xrow[q] = a.Xp[static_cast<int64_t>(row) * a.dk + q];
        __syncthreads();
        unsigned long long L[KP];
#pragma unroll
        for (int p = 0; p < KP; ++p) L[p] = kNoKey;
        for (int j = tid; j < a.m; j += 256) {
            const float4 *yp = reinterpret_cast<const float4 *>(a.Yp + static_cast<int64_t>(j) * a.dk);
            const float4 *xp = reinterpret_cast<const float4 *>(xrow);
            float acc = 0.f;
            for (int q = 0; q < a.dk / 4; ++q) {
                const float4 x = xp[q], y = __ldg(yp + q);
                acc = sqdiff_fma(x.x, y.x, acc);
                acc = sqdiff_fma(x.y, y.y, acc);
                acc = sqdiff_fma(x.z, y.z, acc);
                acc = sqdiff_fma(x.w, y.w, acc);
            }
            const unsigned long long key =
                key64(__fsqrt_rn(acc), static_cast<unsigned>(a.permY ? a.permY[j] : j));
            if (key < L[KP - 1]) {
                L[KP - 1] = key;
#pragma unroll
                for (int p = KP - 1; p > 0; --p) {
                    const unsigned long long lo = min(L[p - 1], L[p]);
                    const unsigned long long hi = max(L[p - 1], L[p]);
                    L[p - 1] = lo;
                    L[p] = hi;
                }
            }
        }
#pragma unroll
        for (int p = 0; p < KP; ++p) lists[tid * KP + p] = L[p];
        __syncthreads();
        // k rounds of a block-wide minimum over the list heads (keys are unique).
        int h = 0;
        for (int p = 0; p < a.k; ++p) {
            const unsigned long long mine = h < KP ? lists[tid * KP + h] : kNoKey;
            unsigned long long m = mine;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = min(m, __shfl_xor_sync(0xffffffffu, m, o));
            if ((tid & 31) == 0) wmin[tid >> 5] = m;
            __syncthreads();
            m = wmin[0];
#pragma unroll
            for (int w = 1; w < 8; ++w) m = min(m, wmin[w]);
            if (mine == m && m != kNoKey) ++h;
            if (tid == 0) {
                const int orow = a.permX ? a.permX[row] : row;
                const int64_t o = static_cast<int64_t>(orow) * a.k + p;
                a.out_idx[o] = static_cast<int32_t>(key_i(m));
                a.out_dist[o] = key_w(m);
                if (a.out_core && p == a.core_rank - 1) a.out_core[orow] = key_w(m);
            }
            __syncthreads();
        }
    }
}

// Split pass of the exact search: item (f, s) is queued row f < rows_cap
// against column range s of `splits`; a block keeps per thread the KP least
// exact (dist, j) keys of its columns (fixed compare-and-swap sink) and writes
// the k least of the block to the item's partial list.
template <int KP>
__global__ void __launch_bounds__(256) knn_exact_split_kernel(const KnnExactArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned long long *lists = reinterpret_cast<unsigned long long *>(smem_raw);  // [256][KP]
    float *xrow = reinterpret_cast<float *>(lists + 256 * KP);                       // [dk]
    __shared__ unsigned long long wmin[8];
    const int tid = threadIdx.x;
    const int rows = min(*a.fb_count, a.rows_cap);
    const int span = (a.m + a.splits - 1) / a.splits;
    for (int item = blockIdx.x; item < rows * a.splits; item += gridDim.x) {
        const int f = item / a.splits, sp = item % a.splits;
        const int row = a.fb_rows[f];
        const int j0 = sp * span, j1 = min(a.m, j0 + span);
        __syncthreads();  // xrow and lists of the previous item are consumed
        for (int q = tid; q < a.dk; q += 256) xrow[q] = a.Xp[static_cast<int64_t>(row) * a.dk + q];
        __syncthreads();
        unsigned long long L[KP];
#pragma unroll
        for (int p = 0; p < KP; ++p) L[p] = kNoKey;
        for (int j = j0 + tid; j < j1; j += 256) {
            const float4 *yp = reinterpret_cast<const float4 *>(a.Yp + static_cast<int64_t>(j) * a.dk);
            const float4 *xp = reinterpret_cast<const float4 *>(xrow);
            float acc = 0.f;
            for (int q = 0; q < a.dk / 4; ++q) {
                const float4 x = xp[q], y = __ldg(yp + q);
                acc = sqdiff_fma(x.x, y.x, acc);
                acc = sqdiff_fma(x.y, y.y, acc);
                acc = sqdiff_fma(x.z, y.z, acc);
                acc = sqdiff_fma(x.w, y.w, acc);
            }
            const unsigned long long key =
                key64(__fsqrt_rn(acc), static_cast<unsigned>(a.permY ? a.permY[j] : j));
            if (key < L[KP - 1]) {
                L[KP - 1] = key;
#pragma unroll
                for (int p = KP - 1; p > 0; --p) {
                    const unsigned long long lo = min(L[p - 1], L[p]);
                    const unsigned long long hi = max(L[p - 1], L[p]);
                    L[p - 1] = lo;
                    L[p] = hi;
                }
            }
        }
#pragma unroll
        for (int p = 0; p < KP; ++p) lists[tid * KP + p] = L[p];
        __syncthreads();
        // k rounds of a block-wide minimum over the list heads (keys are unique)
        int h = 0;
        unsigned long long *out = a.part + static_cast<int64_t>(item) * KP;
        for (int p = 0; p < a.k; ++p) {
            const unsigned long long mine = h < KP ? lists[tid * KP + h] : kNoKey;
            unsigned long long m = mine;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = min(m, __shfl_xor_sync(0xffffffffu, m, o));
            if ((tid & 31) == 0) wmin[tid >> 5] = m;
            __syncthreads();
            m = wmin[0];
#pragma unroll
            for (int w = 1; w < 8; ++w) m = min(m, wmin[w]);
            if (mine == m && m != kNoKey) ++h;
            if (tid == 0) out[p] = m;
            __syncthreads();
        }
    }
}

// Merge pass: one warp per queued row f < rows_cap; lane s walks the sorted
// partial list of split s, and k rounds of a warp minimum pick the row's k
// least keys.
template <int KP>
__global__ void __launch_bounds__(128) knn_exact_merge_kernel(const KnnExactArgs a) {
    const int lane = threadIdx.x & 31;
    const int f = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int rows = min(*a.fb_count, a.rows_cap);
    if (f >= rows) return;
    const int row = a.fb_rows[f];
    const unsigned long long *lst = a.part + (static_cast<int64_t>(f) * a.splits + lane) * KP;
    int h = 0;
    for (int p = 0; p < a.k; ++p) {
        const unsigned long long mine = (lane < a.splits && h < a.k) ? lst[h] : kNoKey;
        unsigned long long m = mine;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = min(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (mine == m && m != kNoKey) ++h;
        if (lane == 0) {
            const int orow = a.permX ? a.permX[row] : row;
            const int64_t o = static_cast<int64_t>(orow) * a.k + p;
            a.out_idx[o] = static_cast<int32_t>(key_i(m));
            a.out_dist[o] = key_w(m);
            if (a.out_core && p == a.core_rank - 1) a.out_core[orow] = key_w(m);
        }
    }
}

template <int KP>
cudaError_t tile_launch(const KnnTileArgs &a, int row_tiles, int splits, cudaStream_t s) {
    const size_t smem = sizeof(TileSmem<KP>);
    cudaError_t e = cudaFuncSetAttribute(knn_tile_kernel<KP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    knn_tile_kernel<KP><<<dim3(row_tiles, splits), kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <int KP>
cudaError_t exact_launch(const KnnExactArgs &a, int blocks, cudaStream_t s) {
    const size_t smem = 256 * KP * sizeof(unsigned long long) + a.dk * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(knn_exact_kernel<KP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(knn_exact_split_kernel<KP>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (a.rows_cap > 0) {
        knn_exact_split_kernel<KP><<<blocks, 256, smem, s>>>(a);
        knn_exact_merge_kernel<KP><<<(a.rows_cap + 3) / 4, 128, 0, s>>>(a);
        count_extra_launches(2);
    }
    knn_exact_kernel<KP><<<blocks, 256, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_knn_tile(int KP, const KnnTileArgs &a, int row_tiles, int splits,
                            cudaStream_t s) {
    if (KP == 16) return tile_launch<16>(a, row_tiles, splits, s);
    if (KP == 32) return tile_launch<32>(a, row_tiles, splits, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_knn_refine(int KP, const KnnRefineArgs &a, int rows, cudaStream_t s) {
    const int per_block = 128 / KP;
    const int blocks = (rows + per_block - 1) / per_block;
    if (KP == 16)
        knn_refine_kernel<16><<<blocks, 128, 0, s>>>(a);
    else if (KP == 32)
        knn_refine_kernel<32><<<blocks, 128, 0, s>>>(a);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_knn_exact(int KP, const KnnExactArgs &a, int blocks, cudaStream_t s) {
    if (KP == 16) return exact_launch<16>(a, blocks, s);
    if (KP == 32) return exact_launch<32>(a, blocks, s);
    return cudaErrorInvalidValue;
}

}  // namespace hdbmst
