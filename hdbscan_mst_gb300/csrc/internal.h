// Host-side launch wrappers of the hdbmst kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <algorithm>
#include <cstddef>
#include <cstdint>

namespace hdbmst {

// ---------------------------------------------------------------- pack.cu
// Copy a caller [d, n] set (leading dim ld) into the padded feature-major
// buffer Xf [dk][n_pad] and, if not nullptr, the point-major buffer
// Xp [n_pad][dk] and, with Xlo, the tensor-core TF32 operand parts
// Xhi = tf32_trunc(x) and Xlo = x - Xhi (both point-major [n_pad][dk], both
// or neither); write
// norm[i] = sum of x^2 (+inf for padding points); flag non-finite values;
// raise *nbmax_bits to the largest norm's bits.  perm (nullable): position
// i < n holds the caller's point perm[i]; or inv (nullable, instead of perm):
// the caller's point i goes to position inv[i] (read in caller order; Xf may
// then be null).  Xh16 / Xl16 (nullable): the
// two-part FP16 operands of the tensor-core tile, point-major [n_pad][dk / 2]
// 32-bit words (two halves each, f16_split with the scale of *amax_bits);
// *e0_out (nullable) then receives the form's absolute error part, rounded up.
// The least squared norm of each 32 consecutive entries of norm[n_pad]
// (n_pad a multiple of 32) into nmin[n_pad / 32].
cudaError_t launch_norm_min32(const float *norm, int64_t n_pad, float *nmin, cudaStream_t s);
cudaError_t launch_pack(const float *X, int64_t ld, int n, int d, int n_pad, int dk, float *Xf,
                        float *Xp, float *Xlo, float *norm, unsigned *status,
                        unsigned *nbmax_bits, cudaStream_t s, const int *perm = nullptr,
                        uint32_t *Xh16 = nullptr, uint32_t *Xl16 = nullptr,
                        const unsigned *amax_bits = nullptr, float *e0_out = nullptr,
                        const int *inv = nullptr, float *Xhi = nullptr);
// Raise *amax_bits to the largest magnitude of a caller [d, n] set.
cudaError_t launch_absmax(const float *X, int64_t ld, int n, int d, unsigned *amax_bits,
                          cudaStream_t s);

// ---------------------------------------------------------------- order.cu
// Spatial order of the tensor-core k-NN (order.cu): nearest of `pivots`
// column points, counting sort by (pivot, bucket of the distance to it), each
// row tile's first column block.
struct SpatialOrder {
    int pivots;              // a multiple of 32
    int buckets;             // distance buckets per pivot cell
    int *cellY, *cellX;      // [m], [n]: bin = cell * buckets + bucket (cellX = cellY when Y is X)
    int *permY, *permX;      // sorted position -> caller index
    int *invY, *invX;        // caller index -> sorted position
    int *startY, *startX;    // [pivots * buckets + 1]: first sorted position of each bin
    int *counters;           // [spatial_counter_ints]
    int *tile_start;         // [row tiles]: first 128-column block of the sweep
    float *pivf;             // [kSpatialMaxD][pivots]: the pivots' features, feature-major
    float *dcellY, *dcellX;  // [m], [n]: distance to the own pivot, caller order
    float *pdY, *pdX;        // nullable, [m][pivots], [n][pivots]: distances to all
                             // pivots, caller order (the pruned search only)
};
inline int spatial_counter_ints(int pivots, int buckets) { return 4 * pivots * buckets + 2 * pivots; }
constexpr int kSpatialMaxD = 192;  // features the spatial order handles (the tensor tile's)
// amax_bits (nullable): raised to the largest finite magnitude of X and Y
// (the FP16 operands' scale), read on the way.
cudaError_t launch_spatial_order(const SpatialOrder &o, const float *X, int64_t ldx, int n,
                                 const float *Y, int64_t ldy, int m, bool alias, int d,
                                 cudaStream_t s, unsigned *amax_bits = nullptr);

// ---------------------------------------------------------------- prune.cu
// Column blocks of the tensor-core k-NN that can hold none of a row tile's
// nearest neighbours, bounded through the pivots of the spatial order.
constexpr int kPrunePivots = 128;   // = SpatialOrder::pivots when pruning
// Blocks of the first pass per row tile: about 1% of the column blocks, 3 to
// kHomeBlocks (200k x 61, of 1, 3, 5, 7, 9, 13, 21 and 31 blocks 13 was
// fastest: a larger home gives the second pass a tighter first threshold).
constexpr int kHomeBlocks = 13;
inline int home_blocks(int col_tiles) {
    const int h = col_tiles / 100;
    return std::min(col_tiles, h < 3 ? 3 : (h > kHomeBlocks ? kHomeBlocks : h));
}
constexpr int kPruneChunks = 4;     // CTAs per row tile in the second pass (at most) when
                                    // its row tiles are not ordered by list length
struct PruneBufs {
    float *Lm, *Hm;       // [P][col_tiles]: per column block, least / largest pivot
                          // distance of its points, widened by the distances' rounding bound
    float2 *HLt;          // [col_tiles][P]: the same (H, L) pairs, block-major
    int *bcell;           // [col_tiles] pivot cell of each block's first point
    float *minH;          // [2 P]: per pivot the least H, then the largest L, over all blocks
    int *home_lo;         // [chunk row tiles] first block of the home range
    int *home;            // [chunk row tiles][kHomeBlocks] home lists
    int *list;            // [chunk row tiles][col_tiles] blocks of the second pass
    int *count;           // [chunk row tiles] entries of list
    int *order;           // [chunk row tiles] row tiles by decreasing count (the second
                          // pass's dispatch order)
    int *slabs;           // [chunk row tiles] partial-list slabs written (1 + chunks)
    unsigned *gthr;       // [chunk rows] shared thresholds of the second pass (KnnTileArgs::gthr)
};
// The column blocks' bounds (from the columns' pivot distances).
cudaError_t launch_prune_setup(const SpatialOrder &o, const PruneBufs &b, int m, int col_tiles,
                               int d, cudaStream_t s);
struct PruneHomeArgs {
    const SpatialOrder *o;
    int n, m, col_tiles, row_tile0, row_tiles;  // row tiles of this chunk: row_tile0 ..
    int nh;                                     // home_blocks(col_tiles)
    bool alias;
};
// Home range of every row tile of a chunk: the kHomeBlocks blocks around the
// columns of the tile's own bin.
cudaError_t launch_prune_home(const PruneHomeArgs &a, const PruneBufs &b, cudaStream_t s);
struct PruneListArgs {
    const float *part_key;  // slab 0: the home pass's sorted lists
    const int *part_idx;
    int chunk_rows_pad, KP, k, d;
    const float *xnorm, *ynorm;  // sorted order
    float err_c;                 // the tile's ranking error coefficient, rounded up
    const float *e0;             // its absolute part (FP16 operands; 0 otherwise)
    int col_tiles, row_base, row_end, row_tiles;
    int chunk_cap;               // blocks per CTA of the second pass
    int nh;                      // blocks of the home range
    unsigned long long *blocks_total;  // += blocks the tile evaluates (both passes)
    const float *pdX;            // [n_pad][P] the rows' pivot distances, callers' order
    const int *permX;            // callers' index of each sorted row position
};
// Upper bound of each row's k-th distance from its home list, the row tile's
// hull per pivot, and the list of blocks that the hull cannot exclude.
cudaError_t launch_prune_lists(const PruneListArgs &a, const PruneBufs &b, cudaStream_t s);
// Row tiles by decreasing list length, ties to the lower tile: order[x] for
// x < row_tiles from count[row_tiles], for at most kOrderMax row tiles.
constexpr int kOrderMax = 8192;
cudaError_t launch_tile_order(const int *count, int row_tiles, int *order, cudaStream_t s);
// Flag core distances that are negative or not finite.
cudaError_t launch_check_core(const float *core, int n, unsigned *status, cudaStream_t s);

// ---------------------------------------------------------------- knn.cu
struct KnnTileArgs {
    const float *Xf;     // [dk][ldx] query rows, feature-major, padded
    const float *Yf;     // [dk][ldy] searched columns, feature-major, padded
    const float *ynorm;  // [ldy] squared norms, +inf past the last column
    const float *ynmin;  // [ldy / 32] least squared norm of each 32 columns (tensor tiles)
    int64_t ldx, ldy;
    int dk;
    int row_base;        // first query row of this chunk
    int row_end;         // one past the last valid query row (n)
    int chunk_rows_pad;  // rows per split slab of the partial lists
    int col_tiles;       // ceil(m / kBN)
    int tiles_per_split;
    float *part_key;     // [S][chunk_rows_pad][KP] approximate keys
    int *part_idx;       // [S][chunk_rows_pad][KP] column indices
    // tensor-core engine only
    const float *Xp, *Yp;  // point-major [.][dk] query rows and columns
    int m;                 // columns
    unsigned *status;      // device status word (timeouts)
    const int *tile_start;  // nullable: per row tile (absolute), first 128-column block of
                            // the sweep, which then wraps around (spatial order)
    // block lists (tensor-core engine, pruned search): the CTA of row tile x
    // (of the chunk) takes blocks blist[x * blist_stride ..], bcount[x] of
    // them (or blist_count when bcount is null), in chunks of chunk_cap, chunk
    // c = gridDim.y - 1 - blockIdx.y, and writes slab slab_base + c
    const int *blist;
    const int *bcount;
    int blist_count, blist_stride, chunk_cap, slab_base;
    const int *tile_order;  // nullable: the row tile of CTA x (longest lists first)
    const float *seed;  // nullable: sorted lists of slab 0 (their KP-th key: a first threshold)
    // nullable (tensor tile, pruned pass): the columns of slab 0's lists; with
    // them every epilogue group's list starts as the row's home list, and the
    // columns of the home range (blocks home_lo[tile] .. + nh - 1) are taken
    // out again before the pass writes its lists (slab 0 holds them)
    const int *seed_idx;
    const int *home_lo;
    int nh;
    // nullable: per row of the chunk, the least KP-th key any CTA of the row's
    // tile holds (float_order bits), read once per tile and lowered with
    // atomicMin: the chunks of one row tile share their thresholds
    unsigned *gthr;
    // tensor-core engine: two-part FP16 operands (dk = 64 only) with the scale of
    // *amax_bits, else three-pass TF32
    int f16;
    const unsigned *amax_bits;
};
// Operands of the tensor-core tiles, point-major: TF32 - a_hi / b_hi the raw
// float32 rows (dk floats), a_lo / b_lo their low parts; FP16 - the hi and lo
// halves (dk / 2 words each).
struct TcOperands {
    const void *a_hi, *a_lo, *b_hi, *b_lo;
};
cudaError_t launch_knn_tile(int KP, const KnnTileArgs &a, int row_tiles, int splits,
                            cudaStream_t s);
// tc_knn.cu: the same tile on tcgen05 TF32 MMAs (three passes), one CTA per SM,
// operands by TMA from the point-major arrays (Xp / Yp and their low parts).
bool tc_knn_supported(int dk);   // dk a multiple of 32, at most kTensorDkMax
bool tc_scan_supported(int dk);  // dk = 32 or 64
cudaError_t launch_tc_knn(int KP, const KnnTileArgs &a, const TcOperands &o, int64_t x_rows,
                          int64_t y_rows, int row_tiles, int splits, cudaStream_t s);
// Test hooks of the tensor-core tiles' failure path, one per translation unit
// (tc.cuh: set_test_hooks), on the current device.
cudaError_t tc_knn_test_hooks(unsigned long long wait_ns, int withhold);
// One CTA: 64 known values per row of 128 TMEM lanes stored and read back
// with the tiles' max-reducing loads; out holds 128 x 68 floats.
cudaError_t tc_tmem_max_probe(float *out, cudaStream_t s);
cudaError_t tc_scan_test_hooks(unsigned long long wait_ns, int withhold);
cudaError_t tc_sym_test_hooks(unsigned long long wait_ns, int withhold);
// Padded feature count: whole 32-feature slabs up to 64 (the tensor-core tile's
// operand granule), multiples of 16 beyond.
// Padded feature count: whole 32-feature slabs up to kTensorDkMax (the
// tensor-core tile works in slabs), else a multiple of 16 (the FFMA tile's K
// step).
constexpr int kTensorDkMax = 192;
inline int padded_features(int d) {
    return d <= kTensorDkMax ? (d + 31) / 32 * 32 : (d + 15) / 16 * 16;
}

struct KnnRefineArgs {
    const float *part_key;
    const int *part_idx;
    int splits, chunk_rows_pad, row_base, row_end;
    const float *Xp, *Yp;  // point-major [.][dk]
    const float *xnorm, *ynorm;
    const unsigned *nbmax_bits;
    float err_c;      // the ranking error is at most err_c (|x|^2 + |y|^2) + *e0
    const float *e0;  // (err_c rounded up; e0 the FP16 operands' absolute part, else 0)
    int d, dk, k, m;
    int core_rank;  // 1-based list position copied to out_core (0: none)
    int32_t *out_idx;
    float *out_dist;
    float *out_core;
    int *fb_count;
    int *fb_rows;
    // spatial order (nullable): caller index of packed row / column positions
    const int *permX, *permY;
    const int *tile_slabs;  // nullable: slabs written per row tile of the chunk (<= splits)
};
cudaError_t launch_knn_refine(int KP, const KnnRefineArgs &a, int rows, cudaStream_t s);

struct KnnExactArgs {
    const int *fb_count;
    const int *fb_rows;
    const float *Xp, *Yp;
    int dk, k, m;
    int core_rank;
    int32_t *out_idx;
    float *out_dist;
    float *out_core;
    // the first rows_cap queued rows are searched with the columns split in
    // `splits` ranges, partial lists in part[(f * splits + s) * KP ..]; any
    // further rows one block per row
    unsigned long long *part;
    int splits, rows_cap;
    const int *permX, *permY;  // as KnnRefineArgs
};
// Exact search of the queued rows: split pass, merge, then the rows beyond
// rows_cap.  blocks: the persistent grid of the split pass and the tail.
cudaError_t launch_knn_exact(int KP, const KnnExactArgs &a, int blocks, cudaStream_t s);

// Launch accounting (api.cu): a wrapper that starts more than one kernel
// reports the kernels beyond the first, which the caller's count covers.
void count_extra_launches(int n);

// ---------------------------------------------------------------- boruvka.cu
cudaError_t launch_mst_init(int n, int *comp, unsigned long long *cand, unsigned long long *ck64,
                            unsigned *chi, unsigned *ub, unsigned long long *cache,
                            cudaStream_t s);
cudaError_t launch_nbr_candidate(int n, int L, const int32_t *kidx, const float *kdist,
                                 const float *core, const int *comp,
                                 const unsigned long long *cache, unsigned long long *cand,
                                 unsigned char *proven, unsigned *ub, unsigned *status,
                                 cudaStream_t s);
cudaError_t launch_classify(int n, const unsigned char *proven, const float *core,
                            const int *comp, const unsigned *ub, unsigned char *act_flag,
                            int *size, int *act_size, int *act_count, cudaStream_t s);
// Slots per component, then the grouped column order (perm and the column
// arrays, col_norm +inf for padding columns) and the active rows grouped by
// component (act_idx).  size, act_size, cursor, act_cursor and totals must
// start at zero.
cudaError_t launch_group(int n, int n_pad, const int *comp, const float *core, const float *norm,
                         const unsigned char *act_flag, const int *size, const int *act_size,
                         int *start, int *act_start, int *cursor, int *act_cursor, int *totals,
                         int *perm, int *col_comp, float *col_core, float *col_norm, int *act_idx,
                         cudaStream_t s);
// Grouped feature-major columns: Xs[f][pos] = Xf[f][perm[pos]] (0 past n).
cudaError_t launch_gather_cols(int n, int n_pad, int dk, const int *perm, const float *Xf,
                               float *Xs, cudaStream_t s);
// Point-major rows by index: dst[r] = src[idx[r]] for r < count, zero up to
// count_pad; both the hi (raw) and lo arrays.
cudaError_t launch_gather_points(int count, int count_pad, int dk, const int *idx,
                                 const float *src_hi, const float *src_lo, float *dst_hi,
                                 float *dst_lo, cudaStream_t s);
cudaError_t launch_gather(int na, int na_pad, int dk, const int *act_idx, const float *Xf,
                          int64_t ldx, const float *core, const int *comp, const float *norm,
                          float *Xa, float *act_core, int *act_comp, float *act_norm,
                          cudaStream_t s);

struct ScanArgs {
    // rows: the active points grouped by component
    const float *Xa;        // [dk][lda] feature-major
    int64_t lda;            // padded active rows (also the stride of the candidate slabs)
    const int *act_idx;     // [na] point index of each active row
    const float *act_core;  // [na]
    const int *act_comp;    // [na]
    const float *act_norm;  // [na] |a|^2
    int na;
    // columns: all points grouped by component
    const float *Xs;        // [dk][ldx] feature-major
    int64_t ldx;
    const int *col_orig;    // [ldx] point index of each column (entries past n unused)
    const float *col_norm;  // [ldx] |b|^2, +inf past the last point
    const float *col_nmin;  // [ldx / 32] least |b|^2 of each 32 columns (tensor scan)
    const float *col_core;  // [ldx] (entries past n unused)
    const int *col_comp;    // [n]
    const int *comp_start;  // [n] first column of each component label
    const int *comp_size;   // [n] columns of each component label
    // by point index (refine and exact search)
    const float *Xp;        // [ldx][dk] point-major
    const float *core;      // [n]
    const int *comp;        // [n]
    const unsigned *nbmax_bits;
    int n, d, dk;
    int col_tiles, tiles_per_split, splits;
    unsigned long long *part_key;  // [splits][lda][4] kept candidates
    float *part_tau;               // [splits][lda] least value of a dropped candidate
    unsigned long long *cand;      // [n] per-point least edge key, lowered by atomicMin
    int *fb_count;
    int *fb_rows;
    unsigned *status;              // device status word (tensor-core timeouts)
    float err_c;                   // ranking error coefficient of the engine that ran (rounded up)
    const float *e0;               // its absolute part (FP16 operands; 0 otherwise)
    int f16;                       // FP16 operands (scale of *amax_bits)
    const unsigned *amax_bits;
    unsigned long long *tile_pairs;  // nullable: += (row, column) pairs the tile evaluates
    // ub (nullable, tensor-core scan): the component bounds U_C; a row then
    // starts from the threshold that U_C implies, and the refine accepts
    // without exactness a row proven to have no edge at or below U_C (it
    // clears the row's act_flag, so the edge is not cached)
    const unsigned *ub;
    unsigned char *act_flag;
};
size_t scan_part_entries(int splits, int64_t lda);
cudaError_t launch_scan(const ScanArgs &a, int row_tiles, int splits, cudaStream_t s);
cudaError_t launch_scan_refine(const ScanArgs &a, cudaStream_t s);
// Rows are the queued points, gathered like the active rows (Xa, act_*, na).
cudaError_t launch_scan_exact(const ScanArgs &a, int row_tiles, int splits, cudaStream_t s);
// tc_scan.cu: the scan on tcgen05 TF32 MMAs; A = active rows, B = grouped
// columns, point-major hi (raw) and lo parts, dk = 32 or 64.
cudaError_t launch_tc_scan(const ScanArgs &a, const float *Xa_hi, const float *Xa_lo,
                           const float *Xs_hi, const float *Xs_lo, int row_tiles, int splits,
                           cudaStream_t s);

// tc_sym.cu: the symmetric scan.  The points of the set P in one order,
// grouped by component, serve as rows and as columns; per component a live
// bound theta (float bits); the pairs that could be a component's cheapest
// edge are recorded as position pairs.
struct SymArgs {
    int np;                  // points in P
    int64_t ld;              // np rounded up to 128 (rows of the operand arrays)
    int blocks;              // ld / 128
    const int *idx;          // [np] point index of each position
    const float *core;       // [ld] core distance by position
    const int *comp;         // [ld] component by position
    const float *norm;       // [ld] |p|^2 by position, +inf past np
    const float *nmin;       // [ld / 32] least |p|^2 of each 32 positions
    const int *comp_start;   // [n] first position of each component label
    const int *comp_size;    // [n] positions of each component label
    const int4 *tile_meta;   // [ld / 64] (component or -1, largest starting bound bits, 0, 0)
    unsigned *theta;         // [n] live bound per component label
    unsigned long long *cand;  // [n] per-point least edge key (weight, other end)
    int2 *pairs;             // [pair_cap] recorded (row, column) positions
    int *pair_count;         // may exceed pair_cap: then the list is incomplete
    int pair_cap;
    int d, dk;
    float err_c;             // ranking error coefficient of the engine (rounded up)
    const float *e0;         // its absolute part
    int f16;
    const unsigned *amax_bits;
    unsigned long long *tile_pairs;
    unsigned *status;
    // nullable: the 128-point blocks of each row tile ([blocks][list_stride],
    // list_count[blocks] entries each) instead of the blocks at or after it
    const int *list;
    const int *list_count;
    int list_stride;
    const int *tile_order;  // nullable: the row tile of CTA x (longest lists first)
};
// The pruned symmetric scan (symprune.cu).  Blocks of 128 positions of P are
// bounded through the pivots of a spatial order of all points; a home pass
// over each row tile's kSymHome nearest blocks (by that bound) of other
// components brings the component bounds close to their final values, and a
// second pass visits the blocks j >= i whose distance bound is at most the
// larger of the two blocks' component bounds.
constexpr int kSymHome = 8;              // blocks per row tile of the home pass
constexpr int kSymMaxComps = 1024;       // components of P the spatial grouping handles
constexpr int kSymChunk = 1024;          // positions of the spatial order per grouping warp
constexpr int kSymPruneMaxBlocks = 8192; // blocks of P (the block-pair arrays are blocks^2)
constexpr int kSymPruneMinN = 16384;     // points below which the scan is not pruned
struct SymPruneBufs {
    SpatialOrder order;  // of all points (X as rows and columns), with pdY [n][128]
    int *kcount;         // [1] compact components assigned
    int *cidx;           // [n] compact index of a component label
    int *cstart;         // [kSymMaxComps] first position of each compact component
    int *off;            // [chunks][kSymMaxComps] counts, then running offsets
    float *Lb, *Hb;      // [blocks][128] least / largest pivot distance per block, widened
    int *bcomp;          // [blocks] component of a block of one component, else -1
    float *LB;           // [blocks][blocks] lower bound of the distance between two blocks
    float *bth;          // [blocks] largest component bound over a block's points
    int *home, *hcount;  // [blocks][kSymHome], [blocks]
    int *hkey;           // [blocks] the home pass's work estimate (larger: more work)
    int *list, *lcount;  // [blocks][blocks], [blocks]
    int *tile_order;     // [blocks] row tiles by decreasing lcount (second pass's dispatch)
};
// P grouped by component in the spatial order (act_idx rewritten): within a
// component, positions follow o.permY.  Needs act_start / act_size of
// launch_group; ncomp <= kSymMaxComps components with points in P.
cudaError_t launch_sym_group(const SymPruneBufs &b, int n, const unsigned char *act_flag,
                             const int *comp, const int *act_start, const int *act_size,
                             int *act_idx, cudaStream_t s);
// Block bounds (Lb, Hb, bcomp), the block-pair bounds LB and the home lists.
cudaError_t launch_sym_blocks(const SymPruneBufs &b, int np, int blocks, const int *act_idx,
                              const int *pcomp, int d, cudaStream_t s);
// After the home pass: bth from the live bounds, and the lists of the second pass.
cudaError_t launch_sym_lists(const SymPruneBufs &b, int np, int blocks, const int *pcomp,
                             const unsigned *theta, int d, cudaStream_t s);
// P = the points with core distance at most the largest U_C over the
// components (act_flag), with per-label counts like launch_classify.
cudaError_t launch_sym_classify(int n, const int *comp, const unsigned *ub, const float *core,
                                unsigned *umax, unsigned char *act_flag, int *size, int *act_size,
                                int *act_count, int *ncomp, cudaStream_t s);
// theta = ub, norm past np = +inf, the tile records.
cudaError_t launch_sym_prepare(int n, int np, int ld, const int *pcomp, const unsigned *ub,
                               unsigned *theta, float *norm, int4 *tile_meta, cudaStream_t s);
cudaError_t launch_tc_sym(const SymArgs &a, const float *x_hi, const float *x_lo, cudaStream_t s);
// The rows the one-sided refine left open against all points on the tensor
// cores (tc_sym.cu): each row's key drops to its exact cheapest edge, the
// columns that need an exact weight appended as point-index pairs.
struct RescanArgs {
    int nr;                   // open rows, gathered (A operand rows nr_pad)
    const int *row_idx;       // [nr] point index
    const float *row_norm;    // [nr_pad] |a|^2
    const float *row_core;    // [nr_pad]
    const int *row_comp;      // [nr_pad]
    int n;                    // columns: all points grouped by component
    int64_t ldx;              // padded columns (rows of the B operand arrays)
    const float *col_norm;    // [ldx] +inf past n
    const float *col_core;    // [ldx]
    const int *col_orig;      // [ldx]
    const int *comp_start, *comp_size;
    int col_tiles, tiles_per_split;
    unsigned long long *cand;
    int2 *pairs;              // [pair_cap] (row point, column point)
    int *pair_count;
    int pair_cap;
    int d, dk;
    float err_c;
    const float *e0;
    int f16;
    const unsigned *amax_bits;
    unsigned *status;
};
cudaError_t launch_tc_rescan(const RescanArgs &a, const float *a_hi, const float *a_lo,
                            const float *b_hi, const float *b_lo, int row_tiles, int splits,
                            cudaStream_t s);
// The recorded pairs' exact weights into both ends' candidate keys (idx null:
// the pairs hold point indices).
cudaError_t launch_sym_pairs_exact(const int2 *pairs, int count, const int *idx, const float *Xp,
                                   int dk, const float *core, unsigned long long *cand,
                                   cudaStream_t s);

// stage 0 also records exact candidates into cache (if not NULL) for the next
// round: the proven ones, and the scanned ones when act_flag is not NULL.
cudaError_t launch_comp_min(int n, const unsigned long long *cand, const int *comp,
                            unsigned long long *ck64, unsigned *chi, const unsigned char *proven,
                            const unsigned char *act_flag, unsigned long long *cache,
                            cudaStream_t s, int stage);
cudaError_t launch_hook(int n, const int *comp, const unsigned long long *ck64,
                        const unsigned *chi, int *parent, int *e_lo, int *e_hi, float *e_w,
                        int *edge_count, unsigned *status, cudaStream_t s);
// Roots of the hook forest by pointer jumping: a first launch and up to
// kJumpMaxLaunches - 1 more, as many as `components` (an upper bound on the
// forest's size) needs (roots_launches); live[kJumpMaxLaunches] holds round
// stamps (any value but `stamp` on entry), so no reset is needed per round.
// relabel sets kStatusNoConverge if a component's pointer did not reach its
// root.
constexpr int kJumpMaxLaunches = 8;  // 16^8 > the largest point count
int roots_launches(int components);
// launch_cap > 0 caps the launches (a test of the bound's detection)
cudaError_t launch_roots(int n, int components, const int *comp, const int *parent, int *root_of,
                         int *live, int stamp, int sms, cudaStream_t s, int launch_cap = 0);
cudaError_t launch_relabel(int n, int *comp, const int *root_of, const int *parent,
                           unsigned long long *cand, unsigned long long *ck64, unsigned *chi,
                           unsigned *ub, unsigned *status, cudaStream_t s);

// ---------------------------------------------------------------- sort.cu
// Sort N edges by (w, lo, hi) ascending and write (lo, hi) pairs and weights.
// tmp buffers hold N entries each; hist holds sort_hist_entries(N) entries
// (three rotating sets of per-tile digit histograms).
size_t sort_hist_entries(int N);
cudaError_t sort_edges(int N, int index_bits, unsigned *w, int *lo, int *hi, unsigned *w2,
                       int *lo2, int *hi2, unsigned *hist, int32_t *out_edges, float *out_w,
                       cudaStream_t s, void (*before)(int, cudaStream_t),
                       void (*after)(int, cudaStream_t));

// ---------------------------------------------------------------- assign.cu
// Bipartite modularity assignment over a k-NN graph (nbr [n, k] int32 indices
// into the m subset points; labels int32 in [0, C)).  degree: right degrees
// (deg_r zeroed by the caller), index checks (kStatusBadList), spikes set to
// -1.  right_mass: K_c of the subset points (zeroes KR first; label checks).
// left: the left step (zeroes KL first, then adds the left masses); *moved
// (zeroed by the caller) counts the spikes that moved.  right: the right step
// (zeroes counts [m][C] first).
cudaError_t launch_assign_degree(const int32_t *nbr, int n, int k, int m, int *deg_r,
                                 int32_t *left, unsigned *status, cudaStream_t s);
cudaError_t launch_assign_right_mass(const int32_t *right, int m, int C, const int *deg_r,
                                     unsigned long long *KR, unsigned *status, cudaStream_t s);
cudaError_t launch_assign_left(const int32_t *nbr, int n, int k, int C, const int32_t *right,
                               const unsigned long long *KR, double gamma, int32_t *left,
                               unsigned long long *KL, int *moved, cudaStream_t s);
cudaError_t launch_assign_right(const int32_t *nbr, int n, int k, int m, int C,
                                const int32_t *left, const int *deg_r,
                                const unsigned long long *KL, double gamma, unsigned *counts,
                                int32_t *right, cudaStream_t s);

// ---------------------------------------------------------------- moments.cu
// Split-product second moment / covariance of a channel-major window.
constexpr int kMomentSplit = 4096;  // samples per split
struct MomentStatus {
    unsigned status;  // kStatus* bits
};
int moment_splits(int64_t n);
// Sub-splits of each split the product takes (a power of two up to 16, so
// that small problems still give about kMomentTargetCtas CTAs); the partial
// products are [splits * sub][c_pad][c_pad].
constexpr int kMomentTargetCtas = 128;
int moment_subsplits(int c_pad, int64_t n);
bool moment_supported();  // the tensor maps the product kernel needs
// stats: channel sums, means (mu_hi + mu_lo) and power-of-two scale
// exponents (scale_e [c_pad], zeroed by the caller for the padding)
cudaError_t launch_moment_stats(const float *X, int64_t ld, int C, int64_t t0, int64_t n,
                                double *sum, float *mu_hi, float *mu_lo, int *scale_e,
                                MomentStatus *st, cudaStream_t s);
// split: the two-part FP16 operands hi, lo [S][c_pad][2048] words of the
// centred window
cudaError_t launch_moment_split(const float *X, int64_t ld, int C, int c_pad, int64_t t0,
                                int64_t n, const float *mu_hi, const float *mu_lo,
                                const int *scale_e, uint32_t *hi, uint32_t *lo, cudaStream_t s);
// product: partial [S][c_pad][c_pad] (upper-triangle 128-tiles) on the tensor cores
cudaError_t launch_moment_product(const uint32_t *hi, const uint32_t *lo, int c_pad, int64_t n,
                                  const int *scale_e, float *partial, unsigned *status,
                                  cudaStream_t s);
// sum: out [C][C] = (or +=) sum over splits / n (+ the centring, uncentred)
cudaError_t launch_moment_sum(const float *partial, int c_pad, int C, int64_t n, int centred,
                              const double *sum, const float *mu_hi, const float *mu_lo,
                              int accumulate, float *out, cudaStream_t s);
cudaError_t moment_test_hooks(unsigned long long wait_ns, int withhold);

// Kernel ids for launch accounting and profiling.
enum KernelId {
    K_PACK = 0,
    K_CHECK_CORE,
    K_KNN_TILE,
    K_KNN_REFINE,
    K_KNN_EXACT,
    K_MST_INIT,
    K_NBR_CANDIDATE,
    K_ACTIVE,
    K_GATHER,
    K_SCAN,
    K_SCAN_REFINE,
    K_SCAN_EXACT,
    K_COMP_MIN,
    K_HOOK,
    K_ROOTS,
    K_RELABEL,
    K_SORT,
    K_PRUNE,
    K_SYM_PRUNE,
    K_ASSIGN_INIT,
    K_ASSIGN_LEFT,
    K_ASSIGN_RIGHT,
    K_MOMENT_PREP,
    K_MOMENT_PRODUCT,
    K_MOMENT_SUM,
    K_COUNT
};

}  // namespace hdbmst
