// K6 in its symmetric form, on the tensor cores: every unordered pair of
// points of different components once, for the rounds in which most points
// need a scan.
//
// Page "HDBSCAN", gpu/hdbscan, "The algorithm on the device": a round needs
// per component only its cheapest edge to another component, and an edge
// (a, b) serves both comp(a) and comp(b).  The one-sided scan (tc_scan.cu)
// visits such an edge twice, once from each end.  Here the points of the set
// P (below) are put in one order, grouped by component, and serve as rows
// and as columns of the same operand arrays; the CTA of row tile i visits the
// 128-point blocks j >= i only (block i included, whose pairs it sees in
// both orientations), skipping the blocks wholly inside its rows' component
// as before.  Each pair is then tested for both ends' components.
//
// Per component C a live bound theta_C (float bits, lowered by atomicMin)
// always weighs at least as much as an edge of C already recorded: it starts
// from the shortcuts' bound U_C (page "HDBSCAN", "Exact shortcuts"; a
// listed edge) and drops to an upper bound of the exact weight of every pair
// recorded.  A pair whose exact weight could be at most theta of either end's
// component is recorded; every other pair provably weighs more than both
// bounds and so more than both components' cheapest edges.  Recording: when
// a core distance is at least the pair's distance bound, the exact weight is
// that core distance and both ends' candidate keys (weight, other end) are
// lowered at once; otherwise the position pair is appended to a list, and
// after the scan sym_pairs_exact_kernel weighs it exactly and lowers both
// keys.  The per-component minimum over the keys is then exactly the
// cheapest edge, ties by (weight, lower, higher) included.
//
// The set P: a pair that could be some component's cheapest edge weighs at
// most that component's bound, so both its cores are at most the largest
// bound; P is the points with core distance at most that (all points when a
// component has no bound).
//
// The test per pair: with t = |b|^2 - 2 a.b from the tile, a pair with
// t >= tau(theta) weighs strictly more than theta (the rounding bound of the engine,
// err_c and e0, and the float32 evaluation of the exact weight; see
// sym_tau), and a pair whose core distances exceed theta does too.  Each
// thread (one row) filters a tile's columns against tau(max(theta_row,
// theta_col)), theta_col the bound of the tile's component (of a tile that
// spans several components, the largest of their starting bounds; a tile
// of two components filters each column range with its own bound).  The
// bounds are read from global memory every few tiles, ahead of their use (a
// column component's first tile waits for its read), so they may be a few
// tiles stale - stale bounds are only larger, and a larger bound only
// records more.  Within a
// 32 x 32 batch the warp first finds the least upper bound of its candidates
// per component and lowers the bounds to it, then records what can still
// win; otherwise every row of every warp would record its own descending
// sequence of improvements.
#include <climits>
#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tc_pipe.cuh"

namespace hdbmst {

namespace {

using namespace tc;

constexpr int kEpiWarps = 12;
constexpr int kSymThreads = (kEpiWarps + 1 + kEpiWarps / 4) * 32;  // + producer + MMA warps

struct TcRescanParams {
    PipeMaps maps;  // B: all points grouped by component, point-major [rows][dk]
    const float *a_hi, *a_lo;  // A: the open rows, point-major
    RescanArgs a;
};

struct TcSymParams {
    PipeMaps maps;  // B: the points of P in grouped order, point-major [rows][dk]
    const float *x_hi, *x_lo;
    SymArgs a;
};

// per warp, two tiles: the columns' norms and core distances, the tile's record
__shared__ float4 s_snorm[kEpiWarps][2][kTileCols / 4];
__shared__ float2 s_snmin[kEpiWarps][2];  // per warp, two tiles: each batch's least norm
__shared__ float4 s_score[kEpiWarps][2][kTileCols / 4];
__shared__ int4 s_smeta[kEpiWarps][2];
constexpr int kListCache = 2048;  // list entries kept in shared memory
__shared__ int s_list[kListCache];

// The filter of a bound th from the row's side (|a|^2 = na): a pair with
// t >= sym_tau(th) weighs strictly more than th.  With th' = max(th, 2^-50)
// and T = th'^2 (1 + 16 u) / (1 - (d + 3) u), a pair's true squared distance
// is at least na + t - c (na + nb) - e0; for nb up to nb_c = (|a| +
// sqrt(T))^2 that exceeds T once t > X = T + c (na + nb_c) + e0 - na, and
// beyond nb_c the distance exceeds sqrt(T) by the triangle inequality.  A
// true squared distance above T (> 2^-100, so no squared difference of it
// underflows) evaluates (float32, ascending features, then sqrt) to more than
// th'.  X is rounded up, plus 2^-20 of its magnitude; the filter is the next
// float above it (t < filter <=> t <= X), so that th = 0 - two copies of a
// point with core distance 0 - still lets equal weights through.
__device__ __forceinline__ float sym_tau(float th, float na, float c, float e0, int d) {
    if (!(th < INFINITY)) return INFINITY;
    const float T = proof_T_up(fmaxf(th, 0x1p-50f), d);
    const float sq = __fadd_ru(__fsqrt_ru(na), __fsqrt_ru(T));
    const float X =
        __fsub_ru(__fadd_ru(__fadd_ru(T, __fmul_ru(c, __fadd_ru(na, __fmul_ru(sq, sq)))), e0), na);
    return nextafterf(__fadd_ru(X, __fmul_ru(__fadd_ru(fabsf(X), __fadd_ru(na, T)), 0x1p-20f)),
                      INFINITY);
}

// An upper bound of the exact weight's distance part from an upper bound D of
// the true squared distance: the float32 sum of d squared differences is at
// most D (1 + (d + 3) u), its correctly rounded square root at most
// sqrt of that times (1 + u); here (1 + 4 u), rounded up.
__device__ __forceinline__ float sym_dist_up(float D, int d) {
    const float m = 1.f + static_cast<float>(d + 4) * 0x1p-24f;
    return __fmul_ru(__fsqrt_ru(__fmul_ru(fmaxf(D, 0.f), m)), 1.f + 0x1p-22f);
}

// A lower bound of the exact weight's distance part from a lower bound D of
// the true squared distance: the float32 sum is at least D (1 - (d + 3) u),
// its square root at least sqrt of that times (1 - u); here (1 - 4 u),
// rounded down.
__device__ __forceinline__ float sym_dist_down(float D, int d) {
    const float m = 1.f - static_cast<float>(d + 4) * 0x1p-24f;
    return __fmul_rd(__fsqrt_rd(__fmul_rd(fmaxf(D, 0.f), m)), 1.f - 0x1p-22f);
}

__device__ __forceinline__ float load_theta(const unsigned *theta, int c) {
    return __uint_as_float(__ldcg(theta + c));
}

// kEW epilogue warps; kSmall: the home pass on the small pipeline (one
// group, a 2-slab ring, 256 TMEM columns), two CTAs per SM.
template <int kEW, bool kSmall>
__global__ void __launch_bounds__((kEW + 1 + kEW / 4) * 32, kSmall ? 2 : 1)
    tc_sym_kernel(const __grid_constant__ TcSymParams P) {
    constexpr int kEpiWarps = kEW;
    extern __shared__ uint8_t smem_raw[];
    __shared__ PipeSmem S;
    __shared__ int s_rcomp[kRows];
    const SymArgs &a = P.a;
    uint8_t *base = pipe_base(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i = a.tile_order ? a.tile_order[blockIdx.x] : static_cast<int>(blockIdx.x);
    const int r0 = i * kRows;
    constexpr int kSub = kCols / kTileCols;

    if (tid < kRows) s_rcomp[tid] = r0 + tid < a.np ? a.comp[r0 + tid] : -1;
    tc_setup<kEpiWarps, false, kSmall>(S);
    fence_before();
    __syncthreads();
    fence_after();
    const bool uniform =
        __syncthreads_and(tid >= kRows || r0 + tid >= a.np || s_rcomp[tid] == s_rcomp[0]);
    int skip_lo = 0, skip_hi = 0;
    if (uniform) {
        const int C = s_rcomp[0];
        const int c0 = a.comp_start[C], c1 = c0 + a.comp_size[C];
        skip_lo = (c0 + kCols - 1) / kCols * kSub;
        skip_hi = c1 / kCols * kSub;
    }
    // the blocks j >= i of the row tile, or its list (cached in shared
    // memory when it fits)
    TileSeq seq(i * kSub, a.blocks * kSub, skip_lo, skip_hi);
    if (a.list) {
        const int cnt = a.list_count[i];
        const int *src = a.list + static_cast<int64_t>(i) * a.list_stride;
        if (cnt <= kListCache) {
            for (int q = tid; q < cnt; q += blockDim.x) s_list[q] = src[q];
            src = s_list;
        }
        seq.list = src;
        seq.n = 2 * cnt;
        __syncthreads();
    }
    if (tid == 0 && a.tile_pairs)
        atomicAdd(a.tile_pairs, static_cast<unsigned long long>(seq.n) * kTileCols * kRows);
    const int dk_mma = a.f16 ? a.dk / 2 : a.dk;
    if (a.f16)
        tc_produce_and_multiply<kEpiWarps, false, true, kSmall>(P.maps, S, smem_u32(base), dk_mma, r0, seq);
    else
        tc_produce_and_multiply<kEpiWarps, false, false, kSmall>(P.maps, S, smem_u32(base), dk_mma, r0, seq);
    if (warp < 4) tc_load_a(S, P.x_hi, P.x_lo, r0, dk_mma);

    if (warp < kEpiWarps) {
        const int row = (warp & 3) * 32 + lane;
        const int r = r0 + row;
        const bool valid = r < a.np;
        const float na = valid ? a.norm[r] : 0.f;
        const float ca = valid ? a.core[r] : INFINITY;
        const int rc = s_rcomp[row];
        const int own_lo = valid ? a.comp_start[rc] : 0;
        const int own_hi = valid ? own_lo + a.comp_size[rc] : 0;
        const float kdot = a.f16 ? -ldexpf(2.f, -2 * f16_scale_exp(*a.amax_bits)) : -2.f;
        const float c = a.err_c, e0 = *a.e0;
        // the row's bound: the value read a few tiles ago, and what this thread recorded
        float pend_r = valid ? load_theta(a.theta, rc) : INFINITY;
        float own_r = INFINITY;
        // the column tile's bound, read one tile ago for component cached_tc
        int cached_tc = -1;
        float pend_c = INFINITY;
        float th_last = -1.f, thr = -INFINITY;

        const auto prefetch = [&](int col0, int buf) {
            static_assert(kTileCols == 64, "one 16-byte copy per lane");
            if (lane < 16) cp_async16(&s_snorm[warp][buf][lane], a.norm + col0 + lane * 4);
            else cp_async16(&s_score[warp][buf][lane - 16], a.core + col0 + (lane - 16) * 4);
            if (lane == 0) cp_async16(&s_smeta[warp][buf], a.tile_meta + col0 / kTileCols);
            if (lane == 1) cp_async8(&s_snmin[warp][buf], a.nmin + (col0 >> 5));
        };
        const auto tau_of = [&](float t) {
            return (!valid || ca > t) ? -INFINITY : sym_tau(t, na, c, e0, a.d);
        };
        // thr = tau(th_last) with th_last >= th: a bound that rose is
        // converted at once; one that dropped keeps the looser filter until
        // it has dropped by 1/256 (the conversion is a chain of correctly
        // rounded square roots and a division)
        const auto retau = [&](float th) {
            if (th > th_last || th < th_last * (1.f - 0x1p-8f)) {
                th_last = th;
                thr = tau_of(th);
            }
        };
        int k_tile = 0;
        tc_epilogue_loop<kEpiWarps, false, kSmall>(S, seq, prefetch, [&](uint32_t tbase, int col0, int buf) {
            // the live bounds are read every 4th tile of the warp (each read
            // is used by the tiles after it; a stale bound is only larger)
            const bool refresh = (k_tile++ & 3) == 0;
            // The tile's columns [0, kb) belong to component c1 with bound
            // th_c, [kb, 64) to c2 with th_c2 (a tile of one component: kb =
            // 64; of three or more: both are the largest starting bound and
            // a candidate reads its own component's bound).
            const int4 meta = s_smeta[warp][buf];
            const int tcomp = meta.x >= 0 ? meta.x : -1;
            const bool two = meta.x < 0 && meta.x >= -kTileCols;
            const int kb = two ? -1 - meta.x : kTileCols;
            float th_c = __int_as_float(meta.y), th_c2 = th_c;
            if (tcomp >= 0) {
                // a new component's bound is read now (once per run of its
                // tiles); later tiles use the value read one tile before
                if (tcomp != cached_tc) {
                    pend_c = load_theta(a.theta, tcomp);
                    cached_tc = tcomp;
                }
                th_c = th_c2 = pend_c;
                if (refresh) pend_c = load_theta(a.theta, tcomp);
            } else if (two) {
                th_c = load_theta(a.theta, meta.z);
                th_c2 = load_theta(a.theta, meta.w);
            }
            float th_r = fminf(pend_r, own_r);
            if (valid && refresh) pend_r = load_theta(a.theta, rc);
            float th = fmaxf(th_r, th_c), th2 = fmaxf(th_r, th_c2);
            retau(th);
            float thr2 = kb < kTileCols ? tau_of(th2) : thr;
            float *nbs = reinterpret_cast<float *>(&s_snorm[warp][buf][0]);
            const float *cbs = reinterpret_cast<const float *>(&s_score[warp][buf][0]);
            // nearly every tile ends here: the floor of each batch's t (its
            // largest dot product against its least norm) reaches the row's
            // filter in every row of the warp; both batches judged after one
            // wait (a batch that passes is loaded again: the accumulator is
            // held until the tile is done)
            float amax0, amax1;
            tmem_ld64_max2(tbase, amax0, amax1);
            const float2 nm2 = s_snmin[warp][buf];
            const unsigned pass =
                (__any_sync(0xffffffffu, batch_t_floor(kdot, amax0, nm2.x) < fmaxf(thr, thr2)) ? 1u : 0u) |
                (__any_sync(0xffffffffu, batch_t_floor(kdot, amax1, nm2.y) < fmaxf(thr, thr2)) ? 2u : 0u);
            if (pass == 0u) return;
#pragma unroll 1
            for (int cc = 0; cc < kTileCols / 32; ++cc) {
                if (!((pass >> cc) & 1u)) continue;
                const int cb0 = col0 + cc * 32;
                const int blo = min(max(own_lo - cb0, 0), 32);
                const int bhi = min(max(own_hi - cb0, 0), 32);
                // tcgen05.ld is warp-collective: skip only what is own for the whole warp
                if (__all_sync(0xffffffffu, blo == 0 && bhi == 32)) continue;
                float v[32];
                tmem_ld32(tbase + cc * 32, v);
                expand32(v, &s_snorm[warp][buf][cc * 8], kdot);
                const float vmin = min32(v);
                const bool hit = vmin < fmaxf(thr, thr2);
                if (!__any_sync(0xffffffffu, hit)) continue;
                const uint32_t own = bhi > blo ? ((bhi == 32 ? 0u : (1u << bhi)) - (1u << blo)) : 0u;
                // columns of this batch in c1's range: bits [0, k1)
                const int k1 = min(max(kb - cc * 32, 0), 32);
                const uint32_t lo_bits = k1 == 32 ? 0xffffffffu : ((1u << k1) - 1u);
                uint32_t mask = 0u;
                if (hit) {
                    mask = below_mask(v, thr) & lo_bits;
                    if (k1 < 32) mask |= below_mask(v, thr2) & ~lo_bits;
                    mask &= ~own;
                }
                // Bounds of a candidate's exact weight, from those of its true
                // squared distance, na + t -/+ (c (na + nb) + e0); its
                // component bc and that component's bound thb; false when its
                // core distances exceed both bounds.
                const auto bounds = [&](int j, float &wlb, float &wub, int &bc, float &thb) -> bool {
                    const bool in1 = cc * 32 + j < kb;
                    const float cm = fmaxf(ca, cbs[cc * 32 + j]);
                    if (cm > (in1 ? th : th2)) return false;
                    const float tj = pick32(v, j);
                    const float err = __fadd_ru(__fmul_ru(c, __fadd_ru(na, nbs[cc * 32 + j])), e0);
                    wub = fmaxf(cm, sym_dist_up(__fadd_ru(__fadd_ru(tj, na), err), a.d));
                    wlb = fmaxf(cm, sym_dist_down(__fsub_rd(__fadd_rd(tj, na), err), a.d));
                    if (tcomp >= 0) {
                        bc = tcomp;
                        thb = th_c;
                    } else if (two) {
                        bc = in1 ? meta.z : meta.w;
                        thb = in1 ? th_c : th_c2;
                    } else {
                        bc = __ldg(a.comp + cb0 + j);
                        thb = load_theta(a.theta, bc);
                    }
                    return true;
                };
                // Pass 1: the least upper bound among the candidates that could
                // be the row component's cheapest edge (best_r), and among
                // those that could be the column's (best_c).
                float best_r = INFINITY, best_c = INFINITY;
                uint32_t keep = 0u;
#pragma unroll 1
                for (uint32_t m = mask; m; m &= m - 1) {
                    const int j = __ffs(m) - 1;
                    if (cb0 + j >= a.np) break;
                    float wlb, wub, thb;
                    int bc;
                    if (!bounds(j, wlb, wub, bc, thb)) continue;
                    const bool for_r = wlb <= th_r, for_c = wlb <= thb;
                    if (!for_r && !for_c) continue;
                    keep |= 1u << j;
                    if (for_r) best_r = fminf(best_r, wub);
                    if (for_c) best_c = fminf(best_c, wub);
                }
                // Over the warp: the least per row component, and (a tile of one
                // component) the least over all rows.  Each least belongs to a
                // pair that pass 2 records, so the bounds may drop to it now.
                const unsigned grp = __match_any_sync(0xffffffffu, rc);
                const float mr = __uint_as_float(__reduce_min_sync(grp, __float_as_uint(best_r)));
                const float mc = tcomp >= 0
                    ? __uint_as_float(__reduce_min_sync(0xffffffffu, __float_as_uint(best_c)))
                    : INFINITY;
                th_r = fminf(th_r, mr);
                own_r = fminf(own_r, mr);
                if (tcomp >= 0) th_c = th_c2 = fminf(th_c, mc);
                // Pass 2: record what can still be either component's cheapest
                // edge.
#pragma unroll 1
                for (uint32_t m = keep; m; m &= m - 1) {
                    const int j = __ffs(m) - 1;
                    const int b = cb0 + j;
                    float wlb, wub, thb;
                    int bc;
                    if (!bounds(j, wlb, wub, bc, thb)) continue;
                    if (!(wlb <= th_r) && !(wlb <= thb)) continue;
                    const float cm = fmaxf(ca, cbs[cc * 32 + j]);
                    if (cm >= wub) {
                        // a core distance dominates: the exact weight is cm, so
                        // both ends' keys are lowered here (equal weights, which
                        // the index order decides, are common in this case)
                        const unsigned ga = static_cast<unsigned>(__ldg(a.idx + r));
                        const unsigned gb = static_cast<unsigned>(__ldg(a.idx + b));
                        atomicMin(a.cand + ga, key64(cm, gb));
                        atomicMin(a.cand + gb, key64(cm, ga));
                    } else {
                        const int pos = atomicAdd(a.pair_count, 1);
                        if (pos >= a.pair_cap) continue;  // the host redoes the round one-sided
                        a.pairs[pos] = make_int2(r, b);
                    }
                    atomicMin(a.theta + rc, __float_as_uint(wub));
                    atomicMin(a.theta + bc, __float_as_uint(wub));
                    own_r = fminf(own_r, wub);
                    th_r = fminf(th_r, wub);
                    if (tcomp >= 0) {
                        th_c = th_c2 = fminf(th_c, wub);
                    } else if (two) {
                        if (cc * 32 + j < kb) th_c = fminf(th_c, wub);
                        else th_c2 = fminf(th_c2, wub);
                    }
                }
                th = fmaxf(th_r, th_c);
                th2 = fmaxf(th_r, th_c2);
                retau(th);
                thr2 = kb < kTileCols ? tau_of(th2) : thr;
            }
        });
    }
    tc_teardown<kEpiWarps, false, kSmall>(S, a.status);
}

// The rows the one-sided refine left open (page "HDBSCAN", "Exact
// shortcuts": only these still lack a proven cheapest edge) against all
// points, on the tensor cores.  Each row starts from th = the exact weight of
// its best kept candidate (its key after the refine, a real edge): a column
// whose weight lower bound (as in the symmetric scan) exceeds th cannot be
// the row's cheapest edge, not even on index order.  A column whose core
// distance dominates its distance bound has that core distance as its exact
// weight and lowers the row's key at once (the ties at the row's own core
// distance - exact copies of the point in other components - that left the
// row open); any other column that can win is appended (point indices) for
// sym_pairs_exact_kernel.  th drops to each recorded column's upper bound.
// Grid: row tiles x column splits.
__shared__ float4 s_rnorm[kEpiWarps][2][kTileCols / 4];
__shared__ float4 s_rcore[kEpiWarps][2][kTileCols / 4];

__global__ void __launch_bounds__(kSymThreads, 1) tc_rescan_kernel(const __grid_constant__ TcRescanParams P) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ PipeSmem S;
    __shared__ int s_rc[kRows];
    const RescanArgs &a = P.a;
    uint8_t *base = pipe_base(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = blockIdx.x * kRows;
    constexpr int kSub = kCols / kTileCols;
    const int ct_begin = blockIdx.y * a.tiles_per_split * kSub;
    const int ct_end = min(blockIdx.y * a.tiles_per_split + a.tiles_per_split, a.col_tiles) * kSub;

    if (tid < kRows) s_rc[tid] = r0 + tid < a.nr ? a.row_comp[r0 + tid] : -1;
    tc_setup<kEpiWarps>(S);
    fence_before();
    __syncthreads();
    fence_after();
    const bool uniform =
        __syncthreads_and(tid >= kRows || r0 + tid >= a.nr || s_rc[tid] == s_rc[0]);
    int skip_lo = 0, skip_hi = 0;
    if (uniform) {
        const int C = s_rc[0];
        const int c0 = a.comp_start[C], c1 = c0 + a.comp_size[C];
        skip_lo = (c0 + kCols - 1) / kCols * kSub;
        skip_hi = c1 / kCols * kSub;
    }
    const TileSeq seq(ct_begin, ct_end, skip_lo, skip_hi);
    const int dk_mma = a.f16 ? a.dk / 2 : a.dk;
    if (a.f16)
        tc_produce_and_multiply<kEpiWarps, false, true>(P.maps, S, smem_u32(base), dk_mma, r0, seq);
    else
        tc_produce_and_multiply<kEpiWarps, false, false>(P.maps, S, smem_u32(base), dk_mma, r0, seq);
    if (warp < 4) tc_load_a(S, P.a_hi, P.a_lo, r0, dk_mma);

    if (warp < kEpiWarps) {
        const int row = (warp & 3) * 32 + lane;
        const int r = r0 + row;
        const bool valid = r < a.nr;
        const float na = valid ? a.row_norm[r] : 0.f;
        const float ca = valid ? a.row_core[r] : INFINITY;
        const int rc = s_rc[row];
        const int ga = valid ? a.row_idx[r] : 0;
        const int own_lo = valid ? a.comp_start[rc] : 0;
        const int own_hi = valid ? own_lo + a.comp_size[rc] : 0;
        const float kdot = a.f16 ? -ldexpf(2.f, -2 * f16_scale_exp(*a.amax_bits)) : -2.f;
        const float c = a.err_c, e0 = *a.e0;
        const unsigned long long k0 = valid ? a.cand[ga] : kNoKey;
        float th = valid ? (k0 == kNoKey ? INFINITY : key_w(k0)) : -INFINITY;
        float thr = valid ? sym_tau(th, na, c, e0, a.d) : -INFINITY;
        const auto prefetch = [&](int col0, int buf) {
            if (lane < 16) cp_async16(&s_rnorm[warp][buf][lane], a.col_norm + col0 + lane * 4);
            else cp_async16(&s_rcore[warp][buf][lane - 16], a.col_core + col0 + (lane - 16) * 4);
        };
        tc_epilogue_loop<kEpiWarps>(S, seq, prefetch, [&](uint32_t tbase, int col0, int buf) {
            const float *nbs = reinterpret_cast<const float *>(&s_rnorm[warp][buf][0]);
            const float *cbs = reinterpret_cast<const float *>(&s_rcore[warp][buf][0]);
#pragma unroll 1
            for (int cc = 0; cc < kTileCols / 32; ++cc) {
                const int cb0 = col0 + cc * 32;
                const int blo = min(max(own_lo - cb0, 0), 32);
                const int bhi = min(max(own_hi - cb0, 0), 32);
                if (__all_sync(0xffffffffu, blo == 0 && bhi == 32)) continue;
                float v[32];
                tmem_ld32(tbase + cc * 32, v);
                expand32(v, &s_rnorm[warp][buf][cc * 8], kdot);
                const float vmin = min32(v);
                // warp-uniform exit: the next batch's TMEM load is collective
                if (!__any_sync(0xffffffffu, vmin < thr)) continue;
                const uint32_t own = bhi > blo ? ((bhi == 32 ? 0u : (1u << bhi)) - (1u << blo)) : 0u;
                uint32_t mask = vmin < thr ? (below_mask(v, thr) & ~own) : 0u;
#pragma unroll 1
                while (mask) {
                    const int j = __ffs(mask) - 1;
                    mask &= mask - 1;
                    const int b = cb0 + j;
                    if (b >= a.n) break;
                    const float cm = fmaxf(ca, cbs[cc * 32 + j]);
                    if (cm > th) continue;
                    const float tj = pick32(v, j);
                    const float err = __fadd_ru(__fmul_ru(c, __fadd_ru(na, nbs[cc * 32 + j])), e0);
                    const float wub = fmaxf(cm, sym_dist_up(__fadd_ru(__fadd_ru(tj, na), err), a.d));
                    const float wlb =
                        fmaxf(cm, sym_dist_down(__fsub_rd(__fadd_rd(tj, na), err), a.d));
                    if (wlb > th) continue;
                    const unsigned gb = static_cast<unsigned>(__ldg(a.col_orig + b));
                    if (cm >= wub) {
                        atomicMin(a.cand + ga, key64(cm, gb));
                    } else {
                        const int pos = atomicAdd(a.pair_count, 1);
                        if (pos >= a.pair_cap) continue;  // the host falls back to the exact scan
                        a.pairs[pos] = make_int2(ga, static_cast<int>(gb));
                    }
                    if (wub < th) {
                        th = wub;
                        thr = sym_tau(th, na, c, e0, a.d);
                    }
                }
            }
        });
    }
    tc_teardown<kEpiWarps>(S, a.status);
}

// Exact weights of the recorded pairs (positions in P, or point indices when
// idx is null), into both ends' candidate keys.  The squared distance is the library's: float32
// differences squared and summed by FMA in ascending feature order.
__global__ void __launch_bounds__(256) sym_pairs_exact_kernel(const int2 *__restrict__ pairs,
                                                              int count,
                                                              const int *__restrict__ idx,
                                                              const float *__restrict__ Xp, int dk,
                                                              const float *__restrict__ core,
                                                              unsigned long long *__restrict__ cand) {
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= count) return;
    const int2 p = pairs[q];
    const int ga = idx ? idx[p.x] : p.x, gb = idx ? idx[p.y] : p.y;
    const float4 *xa = reinterpret_cast<const float4 *>(Xp + static_cast<int64_t>(ga) * dk);
    const float4 *xb = reinterpret_cast<const float4 *>(Xp + static_cast<int64_t>(gb) * dk);
    float acc = 0.f;
    for (int f = 0; f < dk / 4; ++f) {
        const float4 u = __ldg(xa + f), v = __ldg(xb + f);
        acc = sqdiff_fma(u.x, v.x, acc);
        acc = sqdiff_fma(u.y, v.y, acc);
        acc = sqdiff_fma(u.z, v.z, acc);
        acc = sqdiff_fma(u.w, v.w, acc);
    }
    const float w = fmaxf(fmaxf(__ldg(core + ga), __ldg(core + gb)), __fsqrt_rn(acc));
    atomicMin(&cand[ga], key64(w, static_cast<unsigned>(gb)));
    atomicMin(&cand[gb], key64(w, static_cast<unsigned>(ga)));
}

// The largest bound over the components (labels c with comp[c] == c).
__global__ void sym_bound_max_kernel(int n, const int *__restrict__ comp,
                                     const unsigned *__restrict__ ub, unsigned *__restrict__ umax) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    unsigned m = 0u;
    if (c < n && comp[c] == c) m = ub[c];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0 && m) atomicMax(umax, m);
}

// The set P (act_flag), per component its point count and its count in P,
// and the number of components with points in P.
__global__ void sym_classify_kernel(int n, const float *__restrict__ core,
                                    const int *__restrict__ comp, const unsigned *__restrict__ umax,
                                    unsigned char *__restrict__ act_flag, int *__restrict__ size,
                                    int *__restrict__ act_size, int *__restrict__ act_count,
                                    int *__restrict__ ncomp) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31;
    const bool valid = i < n;
    const int cl = valid ? comp[i] : -1;
    const float bound = __uint_as_float(*umax);
    const bool act = valid && core[i] <= bound;
    if (valid) act_flag[i] = act ? 1 : 0;
    const unsigned peers = __match_any_sync(0xffffffffu, cl);
    if (valid && lane == __ffs(peers) - 1) atomicAdd(&size[cl], __popc(peers));
    const unsigned actb = __ballot_sync(0xffffffffu, act);
    const unsigned apeers = peers & actb;
    if (act && lane == __ffs(apeers) - 1 && atomicAdd(&act_size[cl], __popc(apeers)) == 0)
        atomicAdd(ncomp, 1);
    if (lane == 0 && actb) atomicAdd(act_count, __popc(actb));
}

// Before the scan: theta = U_C for every label; the norms past the last
// point of P to +inf (they never rank); per 64-position tile its record
// (x: the component if every point of the tile has the same one, -1 - k if
// the tile holds two, the first on its columns [0, k), -128 for more or for
// padding only; y: the
// largest starting bound over its components; z, w: the first and the second
// component).
__global__ void sym_prepare_kernel(int n, int np, int ld, const int *__restrict__ pcomp,
                                   const unsigned *__restrict__ ub, unsigned *__restrict__ theta,
                                   float *__restrict__ norm, int4 *__restrict__ tile_meta) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) theta[i] = ub[i];
    if (i >= np && i < ld) norm[i] = INFINITY;
    const int t = i;
    if (t < ld / kTileCols) {
        const int p0 = t * kTileCols, p1 = min(p0 + kTileCols, np);
        // components in position order: c1 on [p0, p0 + k), c2 after it
        int c1 = -1, c2 = -1, k = 0, runs = 0;
        unsigned mx = 0u;
        for (int p = p0; p < p1; ++p) {
            const int cp = pcomp[p];
            if (runs == 0 || cp != (runs == 1 ? c1 : c2)) {
                ++runs;
                if (runs == 1) c1 = cp;
                else if (runs == 2) { c2 = cp; k = p - p0; }
            }
            mx = max(mx, ub[cp]);
        }
        int x;
        if (runs == 1) x = c1;              // one component
        else if (runs == 2) x = -1 - k;     // two, split at column k in [1, 63]
        else x = -2 * kTileCols;            // three or more, or padding only
        tile_meta[t] = make_int4(x, static_cast<int>(mx), c1, c2);
    }
}

}  // namespace

cudaError_t launch_sym_classify(int n, const int *comp, const unsigned *ub, const float *core,
                                unsigned *umax, unsigned char *act_flag, int *size, int *act_size,
                                int *act_count, int *ncomp, cudaStream_t s) {
    const int blocks = (n + 255) / 256;
    sym_bound_max_kernel<<<blocks, 256, 0, s>>>(n, comp, ub, umax);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_extra_launches(1);
    sym_classify_kernel<<<blocks, 256, 0, s>>>(n, core, comp, umax, act_flag, size, act_size,
                                               act_count, ncomp);
    return cudaGetLastError();
}

cudaError_t launch_sym_prepare(int n, int np, int ld, const int *pcomp, const unsigned *ub,
                               unsigned *theta, float *norm, int4 *tile_meta, cudaStream_t s) {
    const int m = max(n, ld);
    sym_prepare_kernel<<<(m + 255) / 256, 256, 0, s>>>(n, np, ld, pcomp, ub, theta, norm,
                                                       tile_meta);
    return cudaGetLastError();
}

cudaError_t launch_tc_sym(const SymArgs &a, const float *x_hi, const float *x_lo, cudaStream_t s) {
    TcSymParams P;
    P.a = a;
    P.x_hi = x_hi;
    P.x_lo = x_lo;
    const int dk_mma = a.f16 ? a.dk / 2 : a.dk;
    if ((a.f16 && dk_mma != kSlab) || !make_point_map(&P.maps.b_hi, x_hi, a.ld, dk_mma) ||
        !make_point_map(&P.maps.b_lo, x_lo, a.ld, dk_mma))
        return cudaErrorInvalidValue;
    // the home pass (its short block list) on the small pipeline
    const bool home = a.list_stride == kSymHome;
    auto kern = home ? tc_sym_kernel<4, true> : tc_sym_kernel<kEpiWarps, false>;
    const size_t smem = home ? kSmallPipeSmem : kPipeSmem;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<a.blocks, home ? (4 + 1 + 1) * 32 : kSymThreads, smem, s>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_tc_rescan(const RescanArgs &a, const float *a_hi, const float *a_lo,
                            const float *b_hi, const float *b_lo, int row_tiles, int splits,
                            cudaStream_t s) {
    TcRescanParams P;
    P.a = a;
    P.a_hi = a_hi;
    P.a_lo = a_lo;
    const int dk_mma = a.f16 ? a.dk / 2 : a.dk;
    if ((a.f16 && dk_mma != kSlab) || !make_point_map(&P.maps.b_hi, b_hi, a.ldx, dk_mma) ||
        !make_point_map(&P.maps.b_lo, b_lo, a.ldx, dk_mma))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(tc_rescan_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kPipeSmem));
    if (e != cudaSuccess) return e;
    tc_rescan_kernel<<<dim3(row_tiles, splits), kSymThreads, kPipeSmem, s>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_sym_pairs_exact(const int2 *pairs, int count, const int *idx, const float *Xp,
                                   int dk, const float *core, unsigned long long *cand,
                                   cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    sym_pairs_exact_kernel<<<(count + 255) / 256, 256, 0, s>>>(pairs, count, idx, Xp, dk, core,
                                                               cand);
    return cudaGetLastError();
}

cudaError_t tc_sym_test_hooks(unsigned long long wait_ns, int withhold) {
    return tc::set_test_hooks(wait_ns, withhold);
}

}  // namespace hdbmst
