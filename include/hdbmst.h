/*
 * hdbmst: exact k-nearest neighbours, HDBSCAN core distances and the minimum
 * spanning tree of the mutual-reachability distance, on one GPU (sm_103a).
 *
 * C ABI.  Every entry point takes plain pointers and sizes.  Unless stated
 * otherwise a pointer is a DEVICE pointer, the caller owns every buffer
 * (inputs, outputs and the workspace), and the library allocates no device
 * memory.  Work is queued on `stream`; a call returns once its result is
 * final on that stream (entry points that must read a device status word
 * synchronise the stream before returning, as stated per call).
 *
 * Point sets are float32 and feature-major: a set of n points with d
 * features is a [d, n] array with leading dimension ld >= n, feature f of
 * point i at X[f * ld + i].  X is that set "as stored": a block of points is a
 * transposed view of it and no copy is needed to read it (page "Kilosort4
 * clustering and matching", neuro-kitchen dsp-kitchen gpu/clustering, section
 * "k-nearest neighbours are a matrix product").
 *
 * Distance.  dist(a, b) is the float32 square root of the float32 sum of
 * squared differences, accumulated in ascending feature order with one fused
 * multiply-add per feature.  It is symmetric and every entry point evaluates
 * exactly this function, so equal inputs give equal bits everywhere.
 * Internally the k-NN search ranks candidates by the expansion
 * |x|^2 + |y|^2 - 2 x.y (same page and section) and then re-evaluates the
 * kept candidates with dist(); a per-row error bound proves the kept set holds
 * the true neighbours, and rows it cannot prove are searched again exactly.
 */
#ifndef HDBMST_H_
#define HDBMST_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *hdbmst_stream;

typedef enum {
    HDBMST_OK = 0,
    HDBMST_ERR_ARG = 1,         /* a size, pointer, stride or count is invalid        */
    HDBMST_ERR_UNSUPPORTED = 2, /* valid but beyond the library's limits (k > KMAX ...) */
    HDBMST_ERR_WORKSPACE = 3,   /* workspace NULL, misaligned or smaller than required */
    HDBMST_ERR_NONFINITE = 4,   /* a NaN or infinity in the points or core distances   */
    HDBMST_ERR_NOCONVERGE = 5,  /* Boruvka made no progress in a round (cannot happen   */
                                /* with a consistent weight function; reported, never  */
                                /* looped on)                                          */
    HDBMST_ERR_CUDA = 6,        /* a CUDA runtime call or kernel launch failed         */
    HDBMST_ERR_TOO_LARGE = 7,   /* the problem does not fit hdbmst_knn_noalloc's fixed */
                                /* scratch (HDBMST_NOALLOC_SCRATCH_BYTES)              */
    HDBMST_ERR_TIMEOUT = 8      /* a wait inside a kernel gave up after its bound      */
                                /* (about 1.5 s); the kernel returned, the device      */
                                /* stays usable, the outputs are not valid             */
} hdbmst_status;

/* Largest k for hdbmst_knn, and largest min_samples + 1 for hdbmst_core_distances. */
#define HDBMST_KMAX 32
/* Largest feature count. */
#define HDBMST_DMAX 4096
/* Largest number of points in a set (indices are int32). */
#define HDBMST_NMAX 1073741823LL

typedef enum {
    HDBMST_OP_KNN = 0,
    HDBMST_OP_CORE = 1,
    HDBMST_OP_MST = 2,
    HDBMST_OP_ASSIGN = 3, /* hdbmst_bipartite_assign: d = n_clusters, k = list length */
    HDBMST_OP_MOMENT = 4  /* hdbmst_second_moment: n = samples, d = channels */
} hdbmst_op;

/*
 * Workspace bytes that `op` needs for these sizes (m and k are ignored where
 * they do not apply: CORE takes k = min_samples, MST takes k = the
 * neighbour-list length or 0).  Returns 0 for invalid sizes.  The workspace
 * must be 256-byte aligned; its contents need no initialisation and are
 * garbage afterwards.
 */
size_t hdbmst_workspace_bytes(int op, int64_t n, int64_t m, int d, int k);

/*
 * Exact k-nearest neighbours (page "Kilosort4 clustering and matching",
 * gpu/clustering, section "k-nearest neighbours are a matrix product": the k
 * smallest distances of each row against a set, rows in chunks so scratch
 * stays bounded; equal distances by ascending index as on page "HDBSCAN",
 * gpu/hdbscan, sections "The hang" and "Exact shortcuts").
 *
 *   X [d, n], leading dim ldx >= n: the query points.
 *   Y [d, m], leading dim ldy >= m: the searched points (may alias X).
 *   1 <= k <= min(m, HDBMST_KMAX), 1 <= d <= HDBMST_DMAX.
 *   out_idx  [n, k] int32, row-major: for query i, indices into Y of its k
 *            nearest points ordered by (dist, index); a query that is also in
 *            Y finds itself (distance 0).
 *   out_dist [n, k] float32: dist() of those pairs.
 *   workspace: hdbmst_workspace_bytes(HDBMST_OP_KNN, n, m, d, k) bytes.
 *
 * Errors: ERR_ARG (bad sizes or NULL pointers), ERR_UNSUPPORTED (k or d too
 * large), ERR_WORKSPACE, ERR_NONFINITE (checked on the device; the stream is
 * synchronised once at the end to read it), ERR_CUDA.  Outputs are
 * unspecified after an error.
 */
hdbmst_status hdbmst_knn(const float *X, int64_t ldx, int64_t n, const float *Y, int64_t ldy,
                         int64_t m, int d, int k, int32_t *out_idx, float *out_dist,
                         void *workspace, size_t workspace_bytes, hdbmst_stream stream);

/*
 * HDBSCAN core distances (page "HDBSCAN", gpu/hdbscan, section "The algorithm
 * on the device"): core_i is the distance from point i to its
 * min_samples-th nearest point of X, counting i itself first.
 *
 *   X [d, n], leading dim ldx >= n; 1 <= min_samples <= n,
 *   min_samples + 1 <= HDBMST_KMAX.
 *   out_core     [n] float32.
 *   out_knn_idx  [n, L] int32 or NULL, out_knn_dist [n, L] float32 or NULL,
 *                with L = min(min_samples + 1, n): each point's L nearest
 *                points of X (itself included) as hdbmst_knn returns them.
 *                Keeping one neighbour more than min_samples is what lets
 *                hdbmst_mr_mst prove some cheapest edges without a scan
 *                (same page, section "Exact shortcuts").  Pass both or neither.
 *   workspace: hdbmst_workspace_bytes(HDBMST_OP_CORE, n, 0, d, min_samples).
 *
 * Errors as hdbmst_knn; synchronises the stream once at the end.
 */
hdbmst_status hdbmst_core_distances(const float *X, int64_t ldx, int64_t n, int d,
                                    int min_samples, float *out_core, int32_t *out_knn_idx,
                                    float *out_knn_dist, void *workspace,
                                    size_t workspace_bytes, hdbmst_stream stream);

/*
 * Minimum spanning tree of the mutual-reachability distance
 * w(a, b) = max(core_a, core_b, dist(a, b)) by Boruvka, ties broken by
 * (weight, lower index, higher index) so the tree is unique (page "HDBSCAN",
 * gpu/hdbscan, section "The algorithm on the device").  Each round finds every
 * component's cheapest edge to another component and merges along them.
 *
 *   X [d, n], leading dim ldx >= n.
 *   core [n] float32, finite and >= 0 (normally hdbmst_core_distances' output).
 *   knn_idx [n, L], knn_dist [n, L] (L = knn_len) or both NULL: when given,
 *            the rounds use the two exact shortcuts of section "Exact
 *            shortcuts" (a listed neighbour edge that reaches the point's own
 *            core distance is its cheapest edge when the list provably holds
 *            every point within that distance; a point whose core distance
 *            exceeds its component's lightest neighbour edge is not scanned).
 *            The lists MUST be exact nearest-neighbour lists of X under dist()
 *            ordered by (dist, index), as hdbmst_core_distances writes them;
 *            the tree is the same with or without them.
 *   out_edges [n - 1, 2] int32 (lo, hi) with lo < hi, and out_w [n - 1]
 *            float32 weights, ordered by (w, lo, hi).  n = 1 writes nothing.
 *   workspace: hdbmst_workspace_bytes(HDBMST_OP_MST, n, 0, d, knn_len).
 *
 * The host reads one small status block per Boruvka round (at most
 * ceil(log2 n) + 2 rounds), so this call synchronises the stream each round.
 * The merge runs on the device: each component hooks onto the component at
 * the other end of its cheapest edge, and the roots of the hook forest are
 * found by pointer jumping in a bounded number of launches (16 steps each,
 * as many launches as log16 of the component count needs).  On its first
 * call from a host thread on a device, the call creates a non-blocking side
 * stream and two events for that thread and device (work beside the caller's
 * stream, joined back before the call returns); they are kept for reuse and
 * released when the process exits.
 * Errors: ERR_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_NONFINITE (points or
 * core), ERR_NOCONVERGE, ERR_CUDA.
 */
hdbmst_status hdbmst_mr_mst(const float *X, int64_t ldx, int64_t n, int d, const float *core,
                            const int32_t *knn_idx, const float *knn_dist, int knn_len,
                            int32_t *out_edges, float *out_w, void *workspace,
                            size_t workspace_bytes, hdbmst_stream stream);

/*
 * k-NN for callers that may not allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for users of
 * the library, not for the method.  Some callers cannot call cudaMalloc or
 * hand the library a workspace: a host application that reserved all device
 * memory up front and gives its plugins no allocator, a latency-critical loop
 * where an allocation could synchronise the device, a process under a hard
 * memory quota.  hdbmst_knn_noalloc returns exactly what hdbmst_knn returns
 * (the exact k nearest under dist() in the same order, so the same bits) but
 * takes its scratch from one fixed array of HDBMST_NOALLOC_SCRATCH_BYTES in
 * the library's device image instead of a caller workspace.  To fit that
 * array it searches every column block, without the block pruning hdbmst_knn
 * applies to large sets (which skips only blocks that provably hold none of a
 * row's neighbours), and in smaller row chunks.  The caller still owns X, Y, out_idx and
 * out_dist, with the meaning, layout and limits of hdbmst_knn.
 *
 *  - The array is allocated once per GPU when the library's device code is
 *    loaded there and stays allocated until the process exits.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - Every call on a device uses the same array, so calls whose work overlaps
 *    on the GPU (two streams, or two host threads) race and give wrong
 *    results: serialise them.  The array keeps the last call's contents; the
 *    call clears what must start at zero itself.
 *  - Problems that need more scratch than the array holds return
 *    HDBMST_ERR_TOO_LARGE before any GPU work.  With dk the padded feature
 *    count (round_up(d, 32) up to 192, round_up(d, 16) beyond), the need is
 *    about c * dk * (round_up(n, 128) + round_up(m, 128)) bytes for the packed
 *    copies, c = 12 when d <= 192 (the tensor-core engine's extra low parts)
 *    and 8 otherwise (half that when Y is X), plus 4 bytes per query, 4
 *    bytes per 32 reference points when d <= 192 (each column batch's least
 *    norm) and at least 64 KiB for the neighbour candidates (128 KiB when
 *    k > 12).
 *  - It calls no cudaMalloc, cudaFree or other allocating routine; it
 *    synchronises the stream once at the end, as hdbmst_knn does.
 *
 * Errors: those of hdbmst_knn (except ERR_WORKSPACE), and ERR_TOO_LARGE.
 */
#define HDBMST_NOALLOC_SCRATCH_BYTES (64u << 20)
hdbmst_status hdbmst_knn_noalloc(const float *X, int64_t ldx, int64_t n, const float *Y,
                                 int64_t ldy, int64_t m, int d, int k, int32_t *out_idx,
                                 float *out_dist, hdbmst_stream stream);

/*
 * Bipartite modularity assignment over a k-NN graph (page "Kilosort4
 * clustering and matching", gpu/clustering, section "Assignment in parallel:
 * why the graph is bipartite").  Left nodes are the n spikes, right nodes the
 * m subset points; spike t has one edge to each of the k subset points its
 * list names (as hdbmst_knn writes it against the subset).  Given the right
 * labels, every spike takes its best cluster at once; then, given the spikes'
 * labels, every subset point; alternately.  A node v of degree k_v takes,
 * among its neighbours' labels, the cluster c of largest
 *     2m * n_vc - gamma * (k_v * K_c)
 * with n_vc its edges to nodes labelled c, K_c the degree sum of the OTHER
 * side's nodes labelled c and 2m = 2 n k (the score n_vc - gamma k_v K_c / 2m
 * scaled by 2m), in float64 with the integer product exact, the product with
 * gamma rounded once and the difference rounded once; equal scores go to the
 * lowest label; a subset point no spike lists keeps its label.  A round is a
 * left step and, unless it moved no spike, a right step (the first left step
 * counts every spike as moved); the call stops after the round in which no
 * spike moved, or after max_rounds left steps.
 *
 *   nbr        [n, k] int32, row-major: indices into the subset, in [0, m).
 *   right_init [m] int32: initial labels of the subset points, in
 *              [0, n_clusters) (the page draws them by k-means++ seeding,
 *              which is the caller's); may alias out_right.
 *   out_left   [n] int32, out_right [m] int32: final labels.
 *   gamma      resolution, finite and >= 0; max_rounds 1 ..
 *              HDBMST_ASSIGN_MAX_ROUNDS (the page caps at 200).
 *   out_rounds HOST int or NULL: left steps taken; the moved spikes of each
 *              are in hdbmst_last_assign_moved (the last is 0 when the labels
 *              converged).
 *   workspace: hdbmst_workspace_bytes(HDBMST_OP_ASSIGN, n, m, n_clusters, k)
 *              bytes (about 4 m n_clusters for the right step's counts).
 *
 * Limits: n <= HDBMST_ASSIGN_NMAX (keeps every integer product of the score
 * exact in float64), k <= HDBMST_KMAX, n_clusters <= HDBMST_ASSIGN_CMAX.
 * Synchronises the stream once to check the indices and labels, then once
 * per round to read the moved-spike counter.  Errors: ERR_ARG (sizes, NULL
 * pointers, gamma, an index or initial label out of range), ERR_UNSUPPORTED,
 * ERR_WORKSPACE, ERR_CUDA.
 */
#define HDBMST_ASSIGN_NMAX (1LL << 23)
#define HDBMST_ASSIGN_CMAX 65536
#define HDBMST_ASSIGN_MAX_ROUNDS 1024
hdbmst_status hdbmst_bipartite_assign(const int32_t *nbr, int64_t n, int k, int64_t m,
                                      int n_clusters, double gamma, const int32_t *right_init,
                                      int32_t *out_left, int32_t *out_right, int max_rounds,
                                      int *out_rounds, void *workspace, size_t workspace_bytes,
                                      hdbmst_stream stream);

/* Spikes each left step of the most recent hdbmst_bipartite_assign call moved
 * (up to max_rounds entries; moved may be NULL); returns the number of rounds.
 * Host-side, not thread-safe. */
int hdbmst_last_assign_moved(int64_t *moved, int max_rounds);

/*
 * Split-product second moment and covariance of a window of a channel-major
 * recording (page "Covariance", gpu/covariance, sections "After: split
 * products" and "The bug a test with an odd length found"):
 *     centred != 0:  C = (V - mu)(V - mu)^T / n   (covariance)
 *     centred == 0:  C = V V^T / n                (second moment)
 * with V the window's samples and mu its channel means.  The window is
 * copied, centred, into a split-major buffer of 4 096-sample splits (any
 * start column and any length; the last split is zero-padded), each split's
 * product is taken on the tensor cores (two-part FP16 operands with one
 * power-of-two scale per channel, hi.hi + hi.lo + lo.hi, float32
 * accumulation in runs of 256 samples added in registers, so no single sum
 * adds more than 4 096 products), and the splits are added in float64 in
 * order and divided by n.  The second moment is formed from the centred
 * products plus the means' part, mu_i s_j + mu_j s_i + n mu_i mu_j with
 * s = sum(x) - n mu, in float64: the same value, without the growth of the
 * running sums that raw products with a common offset would have.
 *
 *   X   [channels, ld] float32, row-major (channel c's sample t at
 *       X[c * ld + t]); the window is columns [t0, t0 + n), t0 + n <= ld.
 *   out [channels, channels] float32, row-major, exactly symmetric; written,
 *       or added to when accumulate != 0 (a running sum over windows).
 *   workspace: hdbmst_workspace_bytes(HDBMST_OP_MOMENT, n, 0, channels, 0)
 *       bytes (about 8 bytes per sample and padded channel, plus the split
 *       partials, 4 * splits * round_up(channels, 128)^2 bytes).
 *
 * Limits: 1 <= channels <= HDBMST_DMAX, 1 <= n <= HDBMST_MOMENT_NMAX.
 * Synchronises the stream once at the end to read its status.  Errors:
 * ERR_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_NONFINITE (a NaN or infinity
 * in the window), ERR_TIMEOUT, ERR_CUDA.
 */
#define HDBMST_MOMENT_NMAX (1LL << 30)
hdbmst_status hdbmst_second_moment(const float *X, int64_t ld, int channels, int64_t t0,
                                   int64_t n, int centred, int accumulate, float *out,
                                   void *workspace, size_t workspace_bytes,
                                   hdbmst_stream stream);

/*
 * HDBSCAN labels from the mutual-reachability minimum spanning tree, on the
 * HOST (page "HDBSCAN", gpu/hdbscan, "The algorithm on the device": the
 * hierarchy, its condensed tree and the excess-of-mass selection run on the
 * host; the upstream sorter runs scikit-learn's HDBSCAN, whose definitions
 * are followed).  Single-linkage merge tree of the edges in (w, lo, hi)
 * order, condensed tree for min_cluster_size, stabilities, excess of mass
 * without a single-cluster result, then each point's nearest selected
 * cluster.
 *
 *   edges  [n-1][2] int32 (lo, hi) and w [n-1] float32, HOST memory, as
 *          hdbmst_mr_mst writes them (copy them to the host first);
 *   n      points; min_cluster_size >= 2;
 *   labels [n] int32 out, HOST memory: cluster numbers 0, 1, ... in ascending
 *          order of each cluster's smallest point index, -1 for noise.
 *
 * Linear in n, single-threaded; no CUDA call, no GPU needed.  Errors:
 * ERR_ARG (sizes, NULL pointers, an index out of range, or edges that do not
 * form a spanning tree), ERR_NONFINITE (a weight that is negative, NaN or
 * infinite).  n = 1 gives one noise point.
 */
hdbmst_status hdbmst_hdbscan_labels(const int32_t *edges, const float *w, int64_t n,
                                    int min_cluster_size, int32_t *labels);

/*
 * Distance-tile engine for the k-NN search (hdbmst_knn, hdbmst_knn_noalloc,
 * hdbmst_core_distances) and the Boruvka scan (hdbmst_mr_mst), process-wide,
 * not thread-safe:
 *   HDBMST_ENGINE_AUTO   tensor cores where supported (k-NN and core
 *                        distances: d <= 192; Boruvka scan: d <= 64), else
 *                        FP32 FFMA (the default);
 *   HDBMST_ENGINE_SIMT   FP32 FFMA register-blocked tile everywhere;
 *   HDBMST_ENGINE_TENSOR same as AUTO;
 *   HDBMST_ENGINE_TF32   tensor cores as AUTO, always with TF32 products.
 * The tensor-core tile ranks candidates (tcgen05) with two-part FP16 products
 * (every value, scaled by one power of two per call, split into a high and a
 * low half; hi.hi + hi.lo + lo.hi) where the points have 33 to 64 features
 * (and, for the k-NN, 97 to 128 or 161 to 192), else with three-pass TF32
 * products.  Every engine reports distances and
 * weights re-evaluated exactly with dist() and proves the kept set against
 * its own rounding bound, so results are identical bit for bit whichever
 * engine ran.  Returns the previous setting; unknown values are ignored.
 */
#define HDBMST_ENGINE_AUTO 0
#define HDBMST_ENGINE_SIMT 1
#define HDBMST_ENGINE_TENSOR 2
#define HDBMST_ENGINE_TF32 3
int hdbmst_set_engine(int engine);

/*
 * Form of the Boruvka scan on the tensor cores (hdbmst_mr_mst), process-wide,
 * not thread-safe:
 *   HDBMST_SCAN_AUTO       symmetric in the rounds where at least half the
 *                          points need a scan, one-sided otherwise (default);
 *   HDBMST_SCAN_ONE_SIDED  every scanned point against all points, each
 *                          edge seen from both ends (page "HDBSCAN", "Exact
 *                          shortcuts": the active points are the rows);
 *   HDBMST_SCAN_SYMMETRIC  symmetric in every round that scans.
 * The symmetric form visits each unordered pair of points of different
 * components once and tests it for both components: per component a bound
 * that an already recorded edge meets (the shortcuts' bound to begin with)
 * is lowered by every pair recorded, and a pair is recorded when its exact
 * weight could be at most either bound; the recorded pairs are then weighed
 * exactly.  The tree is the same whichever form runs (the minimum edge per
 * component is exact in both).  With the FP32 FFMA engine, or without
 * nearest lists (no bound), the scan is one-sided.  If a round records more
 * pairs than its list holds, that round is redone one-sided.  Returns the
 * previous setting; unknown values are ignored.
 */
#define HDBMST_SCAN_AUTO 0
#define HDBMST_SCAN_ONE_SIDED 1
#define HDBMST_SCAN_SYMMETRIC 2
int hdbmst_set_scan_form(int form);

/*
 * Block pruning of the symmetric scan (process-wide, not thread-safe; on by
 * default).  It applies with at least 16 384 points, at most 64 features,
 * at most 1024 components with points to scan and at most 8192 blocks of
 * 128 such points.  The points are grouped by component in a spatial order
 * (nearest of 128 pivots, then distance to it); a home pass evaluates each
 * block's 8 nearest blocks of other components (by the pivots'
 * triangle-inequality bound); the second pass skips every block pair whose
 * distance bound exceeds the component bounds the home pass left (page
 * "HDBSCAN", "Exact shortcuts": work is skipped only where a bound proves it
 * cannot change the result).  The tree is the same with it on or off.
 * on = 0 turns it off; returns the previous setting (1 or 0).
 */
int hdbmst_set_scan_pruning(int on);

/*
 * Largest number of pairs the symmetric scan's list (and the list of the
 * open-row rescan, the tensor-core search of the rows the one-sided refine
 * could not prove) may hold; cap <= 0 restores the default (the scratch they
 * reuse, about 32 entries per point).  A round whose list overflows is
 * redone with the one-sided scan, rows whose rescan list overflows are
 * searched by the FP32 exact scan; the tree is the same.  For tests of those
 * fallbacks; process-wide, not thread-safe.  Returns the previous cap (0 for
 * the default).
 */
int64_t hdbmst_set_scan_list_cap(int64_t cap);

/*
 * Test hooks of the failure paths (page "HDBSCAN", gpu/hdbscan, section "The
 * hang": every loop on the device is bounded, and a bound must end in a
 * reported error, not a hang).  They exist so that tests can drive the
 * bounds; leave them off in production.  Both are process-wide and not
 * thread-safe.
 *
 * hdbmst_test_set_tc_hooks: on the CURRENT device, sets how long a wait
 *   inside a tensor-core distance tile may last before it gives up (wait_ns;
 *   0 restores the default of 1.5 s), and, when withhold_first_slab is
 *   non-zero, makes every such tile leave the first slab of its column
 *   stream unloaded.  The tile's waits on that slab then run out: the kernel
 *   winds down, frees its tensor memory and returns, and the call that
 *   launched it returns HDBMST_ERR_TIMEOUT with its outputs invalid; the
 *   device stays usable.  Call (0, 0) to restore.  Synchronous (a small copy
 *   to device memory); returns HDBMST_OK or HDBMST_ERR_CUDA.
 *
 * hdbmst_test_set_mst_caps: caps hdbmst_mr_mst's Boruvka rounds (max_rounds)
 *   and the pointer-jumping launches of each round's merge
 *   (max_jump_launches); 0 means no cap (the default bounds: ceil(log2 n) + 2
 *   rounds, and as many launches of 16-step jumps as the number of
 *   components needs).  A call that runs out of rounds before the tree is
 *   complete, or whose merge leaves a component pointer short of its root,
 *   returns HDBMST_ERR_NOCONVERGE.
 */
hdbmst_status hdbmst_test_set_tc_hooks(uint64_t wait_ns, int withhold_first_slab);

/*
 * hdbmst_test_tmem_max: on the CURRENT device, checks the tensor-memory
 *   load with a max reduction that the tensor-core tiles use to rule out a
 *   32-column batch by the floor of its t (page "Kilosort4 clustering and
 *   matching", "k-nearest neighbours are a matrix product": the batch's
 *   least t is at least its least column norm minus twice its largest dot
 *   product).  One CTA stores 64 known values in each of 128 TMEM lanes and
 *   reads them back as the tiles do; out (device, 128 x 68 floats, row-major)
 *   receives per lane the 64 values read back, then the maxima of columns
 *   0..31 and 32..63 from the one-batch load and from the two-batch load.
 *   The values: ((37 r + 11 c + 5 (r xor c)) mod 97 - 48) * 0.75 for lane r and
 *   column c, except 100 + r at c = r mod 64 and -200 - r at c = (r + 7) mod
 *   64.  Synchronous on the legacy default stream; returns HDBMST_OK,
 *   HDBMST_ERR_ARG (null out) or HDBMST_ERR_CUDA.
 */
hdbmst_status hdbmst_test_tmem_max(float *out);
void hdbmst_test_set_mst_caps(int max_rounds, int max_jump_launches);

/* Human-readable text of a status code (a static string). */
const char *hdbmst_status_string(hdbmst_status status);

/* Name of the CUDA error behind the most recent HDBMST_ERR_CUDA of this
 * process ("cudaSuccess" if there was none); host-side, not thread-safe. */
const char *hdbmst_last_cuda_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int hdbmst_version(void);

/*
 * Instrumentation (host-side, process-wide, not thread-safe).
 *
 * hdbmst_launch_count: kernels this library has launched since load.
 * hdbmst_profile_enable(1): record a CUDA event pair around every kernel
 *   launch, on the launching stream, grouped by kernel; 0 stops recording.
 *   Enabling creates a pool of events on the current device first, so that
 *   no event is created between launches.
 * hdbmst_profile_read: synchronises the recorded events, writes per-kernel
 *   total milliseconds and launch counts for up to max_kernels kernels
 *   (either pointer may be NULL), clears the record and returns the number of
 *   kernels.  hdbmst_profile_kernel_name(i) names entry i.
 */
uint64_t hdbmst_launch_count(void);
void hdbmst_profile_enable(int on);
int hdbmst_profile_read(double *total_ms, int64_t *launches, int max_kernels);
const char *hdbmst_profile_kernel_name(int i);

/*
 * Rows of the most recent hdbmst_knn / hdbmst_knn_noalloc /
 * hdbmst_core_distances call in this process whose candidate set the rounding
 * proof could not close, so that they were searched exactly over all points
 * (host-side, not thread-safe).
 */
int64_t hdbmst_last_knn_exact_rows(void);

/*
 * (row, column) pairs whose distances the distance tile of the most recent
 * hdbmst_knn / hdbmst_knn_noalloc / hdbmst_core_distances call evaluated, in
 * whole blocks of 128 rows x 128 columns (padding included; host-side, not
 * thread-safe).  On the tensor-core path with the spatial order, column blocks
 * that the pivots' triangle-inequality bound proves to hold none of a row
 * block's k nearest are never evaluated (an exact shortcut in the sense of the
 * page "HDBSCAN", section "Exact shortcuts"), so this can be far below n x m.
 */
int64_t hdbmst_last_knn_tile_pairs(void);

/*
 * (row, column) pairs whose distances the Boruvka scan tiles of the most
 * recent hdbmst_mr_mst call evaluated, over all rounds, in whole tiles
 * (padding included; the exact re-scan of rows the rounding proof left open
 * is not counted; host-side, not thread-safe).  Rows are the points the
 * shortcuts of the page "HDBSCAN" ("Exact shortcuts") leave active; tiles
 * wholly inside a row tile's own component are not evaluated.
 */
int64_t hdbmst_last_mst_scan_pairs(void);

/*
 * Rounds of the most recent hdbmst_mr_mst call in this process: returns the
 * number of Boruvka rounds; for each of the first max_rounds rounds writes
 * the number of points scanned against all others (active[i]), the tree
 * edges found so far (edges[i]) and how many scanned points the rounding
 * proof could not settle and were searched again exactly (exact_rows[i]).
 * Any pointer may be NULL.
 */
int hdbmst_last_mst_rounds(int64_t *active, int64_t *edges, int64_t *exact_rows,
                           int max_rounds);

/*
 * Per round of the most recent hdbmst_mr_mst call: the pairs the symmetric
 * scan recorded (recorded[i]), or -1 where the round scanned one-sided (for a
 * symmetric round, active[i] of hdbmst_last_mst_rounds is the size of the
 * set that was scanned).  Returns the number of rounds; recorded may be NULL.
 */
int hdbmst_last_mst_symmetric(int64_t *recorded, int max_rounds);

#ifdef __cplusplus
}
#endif

#endif /* HDBMST_H_ */
