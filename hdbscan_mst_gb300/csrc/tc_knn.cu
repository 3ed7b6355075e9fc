// K1 on the tensor cores: the k-NN distance tile with tcgen05 TF32 MMAs.
//
// Same contract as knn_tile_kernel (page "Kilosort4 clustering and matching",
// gpu/clustering, "k-nearest neighbours are a matrix product": the distances
// of a block of rows to a set are one matrix product plus two norm vectors,
// and a small selection keeps the smallest per row).  A CTA owns 128 query
// rows and a range of 128-column tiles; it writes, per row, the KP best
// (t = |y|^2 - 2 x.y, column) of its range, which knn_refine_kernel merges,
// re-evaluates exactly and proves (with this engine's rounding bound).  The
// pipeline works in 64-column tiles, two per 128-column tile of the split.
//
// Warp roles (one CTA per SM): E epilogue warps (E = 12 for KP = 16 and
// dk <= 64, else 8), then one producer warp and E / 4 MMA warps.  Rows of
// more than 64 padded features (up to 192) use the pipeline's wide variant:
// A hi in TMEM, A lo in shared memory.
//  * the first epilogue group writes the CTA's query rows (hi and lo parts)
//    into TMEM once, where the MMAs read them as the A operand;
//  * the producer (one lane) streams every column tile with TMA slab by slab
//    (32 features, hi and lo) through a 6-stage ring guarded by full/empty
//    mbarriers;
//  * the MMA warps (one lane each, one per group's tiles) issue per slab 3 x 4
//    TF32 MMAs (hi.hi + hi.lo + lo.hi) into the tile's TMEM accumulator, free
//    each ring stage with tcgen05.commit, and signal the accumulator when a
//    tile is complete;
//  * the epilogue warps form E / 4 groups; group g takes every (E / 4)-th
//    tile whole (its two accumulators alternate), and warp w of it reads TMEM
//    lanes 32 (w % 4) .. (its 32 rows), 32 columns at a time.  Each row thus has one list per group, kept
//    in registers by the fixed compare-and-swap sink (page "HDBSCAN", "The
//    hang").  The groups publish each row's KP-th key in shared memory and
//    filter against the least of them (a candidate that cannot beat it cannot
//    reach the row's top KP), so the row's insertions stay close to those of
//    one list.  A warp reads the column norms of a tile from its own shared
//    buffer, filled by cp.async while the tile before was multiplied.  At the
//    end the lists of a row are merged.
// Every wait is bounded; a wait that gives up flags the status word, stops
// every role, drains what it issued, and the CTA frees its TMEM.
#include <climits>
#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tc_pipe.cuh"

namespace hdbmst {

namespace {

using namespace tc;

struct TcKnnParams {
    PipeMaps maps;               // B: columns, point-major [rows][dk]
    const float *a_hi, *a_lo;    // A: query rows, point-major [rows][dk]
    KnnTileArgs a;
};

template <int KP, bool kWide, bool kFill = false>
struct Epi {
    // epilogue warps: 12 (three groups) where the lists are short and the
    // epilogue keeps pace with the products; 8 with more registers each for
    // 32-long lists, wide rows and the home pass (fewer lists to fill)
    // the narrow home pass: one group on the small pipeline, two CTAs per SM
    static constexpr bool kSmall = kFill && !kWide;
    static constexpr int kWarps = kSmall ? 4 : (KP == 16 && !kWide && !kFill) ? 12 : 8;
    static constexpr int kMinBlocks = kSmall ? 2 : 1;
    static constexpr int kParts = kWarps / 4;          // groups: lists per row
    static constexpr int kThreads = (kWarps + 1 + kWarps / 4) * 32;  // + producer + MMA warps
};

__shared__ float g_row_tau[4][kRows];  // per group and row: that list's KP-th key
// per group and row: that list's q-th key, q = ceil(KP / groups): once every
// group holds q keys, their largest q-th key has at least KP keys at or below it
__shared__ float s_row_tq[4][kRows];
// per row: the CTA's threshold, the least of the groups' KP-th keys and the
// largest of their q-th keys, written by the thread that last inserted
// (every value written is a valid bound, so a stale one only loosens it)
__shared__ float s_row_thr[kRows];
// the CTA's block list, when it fits: every role reads it per tile
constexpr int kListCache = 2048;
__shared__ int s_blist[kListCache];
constexpr int kMaxEpiWarps = 12;
__shared__ float4 s_cnorm[kMaxEpiWarps][2][kTileCols / 4];  // per warp: two tiles' column norms
__shared__ float2 s_nmin[kMaxEpiWarps][2];  // per warp, two tiles: each batch's least column norm
// per warp, two tiles: its 32 rows' thresholds shared across CTAs (ordered float bits)
__shared__ uint4 s_gthr[kMaxEpiWarps][2][8];

// A row's list holds (t, column) as one 64-bit key: the order-preserving
// bits of t above the column, so that unsigned order is (t, column) order and
// each compare-and-swap of the fixed sink ("The hang") is one 64-bit minimum
// and maximum (measured: the pruned k-NN tile 5.51 -> 4.50 ms on 200k x 61
// against separate float and index registers; the insertions bound it).
__device__ __forceinline__ unsigned long long pack_tj(float t, int j) {
    return (static_cast<unsigned long long>(float_order(t)) << 32) | static_cast<unsigned>(j);
}
__device__ __forceinline__ float key_t(unsigned long long x) {
    return order_float(static_cast<unsigned>(x >> 32));
}
__device__ __forceinline__ int key_j(unsigned long long x) {
    return static_cast<int>(x & 0xffffffffu);
}

template <int KP>
__device__ __forceinline__ void list_insert(unsigned long long (&k)[KP], unsigned long long x) {
    // keys distinct, k sorted: slot p keeps k[p] if it is below x, else
    // takes x (when k[p - 1] is below x) or k[p - 1]; every slot at once
    bool below[KP];
#pragma unroll
    for (int p = 0; p < KP; ++p) below[p] = k[p] < x;
#pragma unroll
    for (int p = KP - 1; p > 0; --p) k[p] = below[p] ? k[p] : (below[p - 1] ? x : k[p - 1]);
    k[0] = below[0] ? k[0] : x;
}

// k <- the KP least of the two sorted lists k and o (keys are distinct):
// k[p] and o[KP - 1 - p] pair the list with the other reversed, so the KP
// lesser of each pair are exactly the KP least of the union, as a bitonic
// sequence; a bitonic half-cleaner cascade then sorts them.
template <int KP>
__device__ __forceinline__ void list_merge(unsigned long long (&k)[KP],
                                           const unsigned long long (&o)[KP]) {
#pragma unroll
    for (int p = 0; p < KP; ++p) k[p] = min(k[p], o[KP - 1 - p]);
#pragma unroll
    for (int h = KP / 2; h > 0; h >>= 1)
#pragma unroll
        for (int p = 0; p < KP; ++p)
            if ((p & h) == 0) {
                const unsigned long long lo = min(k[p], k[p + h]), hi = max(k[p], k[p + h]);
                k[p] = lo;
                k[p + h] = hi;
            }
}

// k sorted ascending (a bitonic network; no key needs to be distinct).
template <int KP>
__device__ __forceinline__ void list_sort(unsigned long long (&k)[KP]) {
#pragma unroll
    for (int w = 2; w <= KP; w <<= 1)
#pragma unroll
        for (int h = w >> 1; h > 0; h >>= 1)
#pragma unroll
            for (int i = 0; i < KP; ++i) {
                const int l = i ^ h;
                if (l > i) {
                    const bool up = (i & w) == 0;
                    const unsigned long long lo = min(k[i], k[l]), hi = max(k[i], k[l]);
                    k[i] = up ? lo : hi;
                    k[l] = up ? hi : lo;
                }
            }
}

// k[i] for a run-time i (a chain of selects: the list stays in registers)
template <int KP>
__device__ __forceinline__ unsigned long long list_at(const unsigned long long (&k)[KP], int i) {
    unsigned long long r = k[0];
#pragma unroll
    for (int p = 1; p < KP; ++p) r = i == p ? k[p] : r;
    return r;
}

// The 16 least of a 32-column batch (columns in mask, the others absent)
// merged into a 16-long list: a bitonic sort of the batch's 32 keys, then
// list_merge with its first 16.
template <int KP>
__device__ __forceinline__ void batch_merge(unsigned long long (&lk)[KP], const float (&v)[32],
                                            uint32_t mask, int c0) {
    if constexpr (KP == 16) {
        unsigned long long b[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
            b[j] = ((mask >> j) & 1u) ? pack_tj(v[j], c0 + j) : ~0ull;
#pragma unroll
        for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
            for (int h = k >> 1; h > 0; h >>= 1)
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int l = i ^ h;
                    if (l > i) {
                        const bool up = (i & k) == 0;
                        const unsigned long long lo = min(b[i], b[l]), hi = max(b[i], b[l]);
                        b[i] = up ? lo : hi;
                        b[l] = up ? hi : lo;
                    }
                }
        unsigned long long o[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) o[j] = b[j];
        list_merge<16>(lk, o);
    }
}

// kFill: the home pass of the pruned search, whose lists start empty: a
// batch where some row has many candidates is sorted and merged whole
// (batch_merge) instead of inserted one candidate at a time.  A separate
// instance, so that the other passes keep their register allocation.
template <int KP, bool kWide, bool kF16, bool kFill>
__global__ void __launch_bounds__(Epi<KP, kWide, kFill>::kThreads, Epi<KP, kWide, kFill>::kMinBlocks)
    tc_knn_kernel(const __grid_constant__ TcKnnParams P) {
    constexpr int kEpiWarps = Epi<KP, kWide, kFill>::kWarps;
    constexpr int kParts = Epi<KP, kWide, kFill>::kParts;
    constexpr bool kSmall = Epi<KP, kWide, kFill>::kSmall;
    extern __shared__ uint8_t smem_raw[];
    __shared__ PipeSmem S;
    const KnnTileArgs &a = P.a;
    uint8_t *base = pipe_base(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row_tile = a.tile_order ? a.tile_order[blockIdx.x] : static_cast<int>(blockIdx.x);
    int split = blockIdx.y;
    const int r0 = a.row_base + row_tile * kRows;
    constexpr int kSub = kCols / kTileCols;  // pipeline tiles per 128-column tile
    const int ct_begin = split * a.tiles_per_split;
    TileSeq seq(ct_begin * kSub, min(ct_begin + a.tiles_per_split, a.col_tiles) * kSub, 0, 0);
    if (a.tile_start) {  // spatial order: the sweep starts at the rows' own neighbourhood
        seq.rot = a.tile_start[r0 / kRows] * kSub;
        seq.wrap = a.col_tiles * kSub;
    }
    if (a.blist) {
        // pruned search: the CTAs of chunks c >= 1, which only long lists
        // have, are dispatched first (c = gridDim.y - 1 - blockIdx.y); the
        // first of a row tile's CTAs to run takes the list's first range (its
        // nearest blocks), so the threshold it shares tightens early
        const int cnt = a.bcount ? a.bcount[row_tile] : a.blist_count;
        const int c = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);
        const int nch = (cnt + a.chunk_cap - 1) / a.chunk_cap;
        if (c >= nch) return;  // the whole CTA, before any barrier or allocation
        const int begin = (nch - 1 - c) * a.chunk_cap;
        const int len = min(a.chunk_cap, cnt - begin);
        split = a.slab_base + c;
        seq = TileSeq(0, 2 * len, 0, 0);
        const int *gl = a.blist + static_cast<int64_t>(row_tile) * a.blist_stride + begin;
        if (len <= kListCache) {
            for (int i = tid; i < len; i += blockDim.x) s_blist[i] = gl[i];
            seq.list = s_blist;  // visible to all after the barrier below
        } else {
            seq.list = gl;
        }
    }

    for (int i = tid; i < 4 * kRows; i += blockDim.x) {
        (&g_row_tau[0][0])[i] = INFINITY;
        (&s_row_tq[0][0])[i] = INFINITY;
        if (i < kRows) s_row_thr[i] = INFINITY;
    }
    tc_setup<kEpiWarps, kWide, kSmall>(S);
    fence_before();
    __syncthreads();
    fence_after();
    // the MMA operands: dk floats (TF32), or dk / 2 words of two halves (FP16)
    const int dk_mma = kF16 ? a.dk / 2 : a.dk;
    tc_produce_and_multiply<kEpiWarps, kWide, kF16, kSmall>(P.maps, S, smem_u32(base), dk_mma, r0, seq);

    if (warp < 4) tc_load_a<kWide, !kWide || kF16>(S, P.a_hi, P.a_lo, r0, dk_mma);
    if (warp < kEpiWarps) {
        // thread = (row, group): rows 32 (w % 4) + lane, group w / 4
        const int row = (warp & 3) * 32 + lane;
        const int group = warp >> 2;
        unsigned long long lk[KP];  // the row's list, sorted (pack_tj)
#pragma unroll
        for (int p = 0; p < KP; ++p) lk[p] = pack_tj(INFINITY, INT_MAX);
        // Group g's q_g-th key (q_g = KP / groups, one more for the first
        // KP % groups groups: the q_g add up to KP): once every group holds
        // q_g keys, the largest of those keys has at least KP keys of the
        // disjoint lists at or below it.
        const int qg = KP / kParts + (group < KP % kParts ? 1 : 0);
        // The pruned pass: the groups' lists start as the row's home list
        // dealt out (entries g, g + groups, ... to group g: q_g of them), so
        // that bound is the home list's KP-th key from the first tile on and
        // drops with every insertion.
        const bool seeded = a.seed_idx != nullptr;
        if (seeded && r0 + row < a.row_end) {
            const int64_t so = static_cast<int64_t>(row_tile * kRows + row) * KP;
#pragma unroll
            for (int p = 0; p < KP; ++p) {
                const int e = group + p * kParts;
                if (e < KP) lk[p] = pack_tj(a.seed[so + e], a.seed_idx[so + e]);
            }
            s_row_tq[group][row] = key_t(list_at(lk, qg - 1));
        }
        // a first threshold: the KP-th key an earlier pass already holds for
        // the row (a candidate at or above it cannot reach the merged top KP)
        float seed = INFINITY;
        if (a.seed && r0 + row < a.row_end)
            seed = a.seed[static_cast<int64_t>(row_tile * kRows + row) * KP + KP - 1];
        unsigned published = 0xffffffffu;  // the least threshold this thread put in gthr
        // t = |y|^2 - 2 x.y; the FP16 products carry the set's scale 2^2e
        const float kdot = kF16 ? -ldexpf(2.f, -2 * f16_scale_exp(*a.amax_bits)) : -2.f;
        // the warp's 32 rows of the shared thresholds (pruned second pass)
        const int local_row = row_tile * kRows + row;
        const unsigned *gthr_warp = a.gthr ? a.gthr + row_tile * kRows + (warp & 3) * 32 : nullptr;
        const auto prefetch = [&](int col0, int buf) {
            if (lane < kTileCols / 4) cp_async16(&s_cnorm[warp][buf][lane], a.ynorm + col0 + lane * 4);
            else if (gthr_warp && lane < kTileCols / 4 + 8)
                cp_async16(&s_gthr[warp][buf][lane - kTileCols / 4], gthr_warp + (lane - kTileCols / 4) * 4);
            else if (lane == 31)
                cp_async8(&s_nmin[warp][buf], a.ynmin + (col0 >> 5));
        };
        float own = key_t(lk[KP - 1]);  // this list's KP-th key
        tc_epilogue_loop<kEpiWarps, kWide, kSmall>(S, seq, prefetch, [&](uint32_t tbase, int col0, int buf) {
            // the seed and the least KP-th key any CTA of the row tile has
            // published (read once per tile)
            const float tile_thr =
                gthr_warp ? fminf(seed, order_float(reinterpret_cast<const unsigned *>(&s_gthr[warp][buf][0])[lane]))
                          : seed;
#pragma unroll 1
            for (int cc = 0; cc < kTileCols / 32; ++cc) {
                float v[32];
                const float amax = tmem_ld32_max(tbase + cc * 32, v);
                // the least of: this list's KP-th key, the CTA's threshold,
                // the seed and the shared threshold
                const float tau = fminf(fminf(own, tile_thr), s_row_thr[row]);
                // most batches end here: their floor of t (the largest dot
                // product against the least norm) reaches every row's threshold
                const float nmin = cc ? s_nmin[warp][buf].y : s_nmin[warp][buf].x;
                if (!__any_sync(0xffffffffu, batch_t_floor(kdot, amax, nmin) < tau)) continue;
                expand32(v, &s_cnorm[warp][buf][cc * 8], kdot);
                // the batch's least t by a depth-5 tree, against the least
                // published KP-th key of the row (stale values only loosen it)
                const float vmin = min32(v);
                if (vmin < tau) {
                    // rare: insert this batch's candidates in column order
                    // with the one copy of the sink
                    uint32_t mask = below_mask(v, tau);
                    if (kFill && __any_sync(__activemask(), __popc(mask) > 14)) {
                        // many candidates (a list still filling): sort the
                        // batch's keys and merge its 16 least into the list
                        batch_merge(lk, v, mask, col0 + cc * 32);
                    } else {
#pragma unroll 1
                        while (mask) {
                            const int j = __ffs(mask) - 1;
                            mask &= mask - 1;
                            list_insert<KP>(lk, pack_tj(pick32(v, j), col0 + cc * 32 + j));
                        }
                    }
                    own = key_t(lk[KP - 1]);
                    g_row_tau[group][row] = own;
                    s_row_tq[group][row] = key_t(list_at(lk, qg - 1));
                    // the CTA's threshold for this row: the least KP-th key
                    // and the largest q_g-th key of the groups' lists
                    float tc = own, tm = -INFINITY;
#pragma unroll
                    for (int q = 0; q < kParts; ++q) {
                        tc = fminf(tc, g_row_tau[q][row]);
                        tm = fmaxf(tm, s_row_tq[q][row]);
                    }
                    const float cta = fminf(tc, tm);
                    s_row_thr[row] = cta;
                    if (gthr_warp && r0 + row < a.row_end) {
                        // for the other CTAs of the row tile
                        const unsigned o = float_order(cta);
                        if (o < published && cta < INFINITY) {
                            published = o;
                            atomicMin(a.gthr + local_row, o);
                        }
                    }
                }
            }
        });
        // the home range's columns leave the lists again (slab 0 holds them)
        if (seeded) {
            const int h0 = a.home_lo[row_tile];
#pragma unroll
            for (int p = 0; p < KP; ++p) {
                const int blk = key_j(lk[p]) / kCols;
                if (blk >= h0 && blk < h0 + a.nh) lk[p] = pack_tj(INFINITY, INT_MAX);
            }
            list_sort<KP>(lk);
        }
        // merge the row's lists: the ring is idle now, other groups park there
        if (kParts > 1) {
            float *pk = reinterpret_cast<float *>(base);
            int *pi = reinterpret_cast<int *>(pk + (kParts - 1) * kRows * KP);
            epilogue_sync<kEpiWarps>();  // every MMA has been consumed
            if (group > 0) {
#pragma unroll
                for (int p = 0; p < KP; ++p) {
                    pk[((group - 1) * kRows + row) * KP + p] = key_t(lk[p]);
                    pi[((group - 1) * kRows + row) * KP + p] = key_j(lk[p]);
                }
            }
            epilogue_sync<kEpiWarps>();
            if (group == 0) {
#pragma unroll 1
                for (int q = 1; q < kParts; ++q) {
                    unsigned long long o[KP];
#pragma unroll
                    for (int p = 0; p < KP; ++p)
                        o[p] = pack_tj(pk[((q - 1) * kRows + row) * KP + p],
                                       pi[((q - 1) * kRows + row) * KP + p]);
                    list_merge<KP>(lk, o);
                }
            }
        }
        if (group == 0 && !*(volatile int *)&S.abort && r0 + row < a.row_end) {
            const int local = row_tile * kRows + row;
            const int64_t o = (static_cast<int64_t>(split) * a.chunk_rows_pad + local) * KP;
#pragma unroll
            for (int p = 0; p < KP; ++p) {
                a.part_key[o + p] = key_t(lk[p]);
                a.part_idx[o + p] = key_j(lk[p]);
            }
        }
    }
    tc_teardown<kEpiWarps, kWide, kSmall>(S, a.status);
}

template <int KP, bool kWide, bool kF16>
cudaError_t tc_launch(const TcKnnParams &P, int row_tiles, int splits, cudaStream_t s) {
    // the home pass of the pruned search: a block list and no seed
    const bool fill = KP == 16 && P.a.blist != nullptr && P.a.seed == nullptr;
    const size_t smem = kWide ? kWidePipeSmem : (fill ? kSmallPipeSmem : kPipeSmem);
    auto kern = fill ? tc_knn_kernel<KP, kWide, kF16, KP == 16> : tc_knn_kernel<KP, kWide, kF16, false>;
    const int threads = fill ? Epi<KP, kWide, KP == 16>::kThreads : Epi<KP, kWide, false>::kThreads;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<dim3(row_tiles, splits), threads, smem, s>>>(P);
    return cudaGetLastError();
}

}  // namespace

bool tc_knn_supported(int dk) {
    static_assert(kWideDkMax == kTensorDkMax, "the packed low parts cover the wide tile");
    return dk % kSlab == 0 && dk >= kSlab && dk <= kWideDkMax && tensor_maps_available();
}

cudaError_t launch_tc_knn(int KP, const KnnTileArgs &a, const TcOperands &o, int64_t x_rows,
                          int64_t y_rows, int row_tiles, int splits, cudaStream_t s) {
    TcKnnParams P;
    P.a = a;
    // the pipeline moves 32-bit words: floats (TF32) or pairs of halves (FP16)
    P.a_hi = static_cast<const float *>(o.a_hi);
    P.a_lo = static_cast<const float *>(o.a_lo);
    const float *b_hi = static_cast<const float *>(o.b_hi), *b_lo = static_cast<const float *>(o.b_lo);
    const bool wide = a.dk > 64;
    // FP16: dk / 2 words of two halves, whole 32-word slabs (dk = 64, 128 or
    // 192); past 64 features both A parts sit in TMEM [0, dk) below the wide
    // layout's accumulators
    const int dk_mma = a.f16 ? a.dk / 2 : a.dk;
    if ((a.f16 && dk_mma % kSlab != 0) || !make_point_map(&P.maps.b_hi, b_hi, y_rows, dk_mma) ||
        !make_point_map(&P.maps.b_lo, b_lo, y_rows, dk_mma) ||
        (wide && !a.f16 && !make_point_map(&P.maps.a_lo, P.a_lo, x_rows, a.dk)))
        return cudaErrorInvalidValue;
    if (a.f16 && !wide && KP == 16) return tc_launch<16, false, true>(P, row_tiles, splits, s);
    if (a.f16 && !wide && KP == 32) return tc_launch<32, false, true>(P, row_tiles, splits, s);
    if (a.f16 && wide && KP == 16) return tc_launch<16, true, true>(P, row_tiles, splits, s);
    if (a.f16 && wide && KP == 32) return tc_launch<32, true, true>(P, row_tiles, splits, s);
    if (!wide && KP == 16) return tc_launch<16, false, false>(P, row_tiles, splits, s);
    if (!wide && KP == 32) return tc_launch<32, false, false>(P, row_tiles, splits, s);
    if (wide && KP == 16) return tc_launch<16, true, false>(P, row_tiles, splits, s);
    if (wide && KP == 32) return tc_launch<32, true, false>(P, row_tiles, splits, s);
    return cudaErrorInvalidValue;
}

// Check of the TMEM loads' max reduction that the tiles' batch floor rests
// on: one CTA of 128 threads allocates 64 TMEM columns, each warp stores 64
// known values per row of its 32 lanes, and the row's values and maxima come
// back as the tiles read them (tmem_ld32_max per 32-column batch, and
// tmem_ld64_max2 for both).  out[row * 68 + c]: the 64 values, then the two
// batch maxima of each form.  The values: ((37 r + 11 c + 5 (r ^ c)) mod 97 -
// 48) * 0.75, except 100 + r at c = r mod 64 and -200 - r at c = (r + 7) mod
// 64 (a unique largest and least value per row).
__global__ void __launch_bounds__(128) tmem_max_probe_kernel(float *out) {
    __shared__ uint32_t s_base;
    const int warp = threadIdx.x >> 5, row = threadIdx.x;
    if (warp == 0) tmem_alloc(&s_base, 64);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t taddr = s_base + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float w[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int c = 32 * h + j;
            float x = static_cast<float>((37 * row + 11 * c + 5 * (row ^ c)) % 97 - 48) * 0.75f;
            if (c == row % 64) x = 100.f + static_cast<float>(row);
            if (c == (row + 7) % 64) x = -200.f - static_cast<float>(row);
            w[j] = x;
        }
        tmem_st32(taddr + 32 * h, w);
    }
    tmem_wait_st();
    float v[32];
    const float m0 = tmem_ld32_max(taddr, v);
    for (int j = 0; j < 32; ++j) out[row * 68 + j] = v[j];
    const float m1 = tmem_ld32_max(taddr + 32, v);
    for (int j = 0; j < 32; ++j) out[row * 68 + 32 + j] = v[j];
    float p0, p1;
    tmem_ld64_max2(taddr, p0, p1);
    out[row * 68 + 64] = m0;
    out[row * 68 + 65] = m1;
    out[row * 68 + 66] = p0;
    out[row * 68 + 67] = p1;
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_free(s_base, 64);
}

cudaError_t tc_tmem_max_probe(float *out, cudaStream_t s) {
    if (!out) return cudaErrorInvalidValue;
    tmem_max_probe_kernel<<<1, 128, 0, s>>>(out);
    return cudaGetLastError();
}

cudaError_t tc_knn_test_hooks(unsigned long long wait_ns, int withhold) {
    return tc::set_test_hooks(wait_ns, withhold);
}

}  // namespace hdbmst
