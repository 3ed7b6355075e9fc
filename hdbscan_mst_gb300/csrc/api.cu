// C ABI of the hdbmst library: argument checks, workspace layout, the
// host-side sequencing of the kernels, and launch accounting.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/hdbmst.h"
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

using namespace hdbmst;

namespace {

// ------------------------------------------------------------------ accounting

std::atomic<uint64_t> g_launches{0};
bool g_prof = false;
struct ProfRec {
    int id;
    cudaEvent_t a, b;
};
std::vector<ProfRec> g_recs;
std::vector<cudaEvent_t> g_pool;
// distance-tile engine (HDBMST_ENGINE_*), process-wide
int g_engine = HDBMST_ENGINE_AUTO;

bool use_tensor(int dk) {
    return g_engine != HDBMST_ENGINE_SIMT && tc_knn_supported(dk);
}

bool use_tensor_scan(int dk) {
    return g_engine != HDBMST_ENGINE_SIMT && tc_scan_supported(dk);
}

// Two-part FP16 operands on the tensor cores: 64 padded features (one
// 128-byte row of halves per part), unless TF32 is asked for.
// The two-part FP16 form: 64 padded features, and (the k-NN tile's wide
// rows) 128 or 192; other widths stay on three-pass TF32.
bool use_f16(int dk) {
    return g_engine != HDBMST_ENGINE_TF32 && (dk == 64 || dk == 128 || dk == 192);
}

// Form of the Boruvka scan on the tensor cores (HDBMST_SCAN_*), process-wide,
// and whether the symmetric form prunes block pairs.
int g_scan_form = HDBMST_SCAN_AUTO;
bool g_sym_prune = true;
// Test caps of hdbmst_mr_mst (0: none): Boruvka rounds, and launches of the
// merge's pointer jumping per round (hdbmst_test_set_mst_caps).
int g_test_max_rounds = 0;
int g_test_jump_launches = 0;
// Cap on the recorded-pair lists of the symmetric scan and of the open-row
// rescan (0: the whole scratch they use); a list that overflows sends its
// round to the one-sided scan, or its rows to the FP32 exact scan.
int64_t g_list_cap = 0;
int list_cap(size_t scratch_pairs) {
    size_t cap = std::min<size_t>(scratch_pairs, 1u << 30);
    if (g_list_cap > 0) cap = std::min<size_t>(cap, static_cast<size_t>(g_list_cap));
    return static_cast<int>(cap);
}

// per-round record of the last hdbmst_mr_mst call: points scanned, edges so
// far, rows searched exactly, pairs the symmetric scan recorded (-1: one-sided)
std::vector<int64_t> g_round_active, g_round_edges, g_round_exact, g_round_sym;
// rows of the last k-NN / core-distance call searched exactly
int64_t g_knn_exact_rows = 0;
// (row, column) pairs the distance tile of the last k-NN / core-distance call
// evaluated, in whole 128 x 128 blocks
int64_t g_knn_tile_pairs = 0;
// (row, column) pairs the Boruvka scan tiles of the last mr_mst call evaluated
int64_t g_mst_scan_pairs = 0;

const char *const kKernelNames[K_COUNT] = {
    "pack",   "check_core", "knn_tile", "knn_refine", "knn_exact", "mst_init",
    "nbr_candidate", "active", "gather", "boruvka_scan", "boruvka_refine", "boruvka_exact",
    "comp_min", "hook",
    "roots",  "relabel",    "sort_edges", "knn_prune", "mst_prune", "assign_init",
    "assign_left", "assign_right", "moment_prep", "moment_product", "moment_sum"};

cudaEvent_t take_event() {
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

void before(int id, cudaStream_t s) {
    if (!g_prof) return;
    ProfRec r{id, take_event(), nullptr};
    cudaEventRecord(r.a, s);
    g_recs.push_back(r);
}

void after(int id, cudaStream_t s) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (!g_prof || g_recs.empty()) return;
    ProfRec &r = g_recs.back();
    if (r.id != id || r.b) return;
    r.b = take_event();
    cudaEventRecord(r.b, s);
}

cudaError_t g_last_cuda = cudaSuccess;

}  // namespace

void hdbmst::count_extra_launches(int n) {
    g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed);
}

namespace {

hdbmst_status cuda_fail(cudaError_t e) {
    g_last_cuda = e;
    return HDBMST_ERR_CUDA;
}

#define LAUNCH(id, stream, call)                         \
    do {                                                 \
        before(id, stream);                              \
        cudaError_t e_ = (call);                         \
        after(id, stream);                               \
        if (e_ != cudaSuccess) return cuda_fail(e_);     \
    } while (0)

#define CUDA_OK(call)                                    \
    do {                                                 \
        cudaError_t e_ = (call);                         \
        if (e_ != cudaSuccess) return cuda_fail(e_);     \
    } while (0)

// ------------------------------------------------------------------ workspace

struct Carver {
    char *base;
    size_t off = 0;
    explicit Carver(void *b) : base(static_cast<char *>(b)) {}
    template <class T>
    T *take(size_t count) {
        off = static_cast<size_t>(round_up(static_cast<int64_t>(off), 256));
        T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
        off += count * sizeof(T);
        return p;
    }
};

struct DevStatus {
    unsigned status;
    unsigned nbmax_bits;
    int fb_count;
    int act_count;
    int edge_count;
    unsigned amax_bits;              // largest magnitude of the points (FP16 operands' scale)
    float e0;                        // the FP16 form's absolute ranking error (0 otherwise)
    unsigned long long tile_blocks;  // 128 x 128 blocks the pruned k-NN tile evaluated
    unsigned long long scan_pairs;   // (row, column) pairs the Boruvka scan evaluated
    unsigned sym_umax;               // symmetric scan: the largest component bound
    int sym_pairs;                   // symmetric scan: pairs recorded (may exceed the list)
    int sym_ncomp;                   // symmetric scan: components with points in P
    int jump_live[kJumpMaxLaunches]; // merge: round stamps of the pointer-jumping launches
};

// A ranking error coefficient as the float32 the proofs use, rounded up.
float coef_up(double c) {
    float f = static_cast<float>(c);
    if (static_cast<double>(f) < c) f = std::nextafter(f, INFINITY);
    return f;
}

constexpr int kMaxSplits = 8;
constexpr int kScanMaxSplits = 16;  // column splits of the one-sided tensor scan (few rows)
constexpr size_t kPartialBudget = size_t(256) << 20;  // bytes of partial lists per chunk

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return 148;
    return sms;
}

// A second stream (per host thread and device) for work that can run beside
// the caller's stream, with the events that fork it from and join it to
// that stream.
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
cudaError_t side_stream(SideStream **out) {
    constexpr int kMaxDevices = 64;
    thread_local SideStream side[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    SideStream &x = side[dev];
    if (!x.s) {
        if ((e = cudaStreamCreateWithFlags(&x.s, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    *out = &x;
    return cudaSuccess;
}

// Makes the caller's stream wait for the side stream's work when it goes out
// of scope (every return path), so no work on the workspace outlives a call.
struct JoinOnExit {
    cudaStream_t s;
    cudaEvent_t e = nullptr;
    ~JoinOnExit() {
        if (e) cudaStreamWaitEvent(s, e, 0);
    }
};

// Column splits that fill the GPU's CTA slots in whole waves.
int choose_splits(int row_tiles, int col_tiles, int slots) {
    int best = 1;
    double best_eff = 0.0;
    const int smax = std::max(1, std::min(kMaxSplits, col_tiles));
    for (int S = 1; S <= smax; ++S) {
        const int64_t units = static_cast<int64_t>(row_tiles) * S;
        const int64_t waves = (units + slots - 1) / slots;
        const double eff = static_cast<double>(units) / static_cast<double>(waves * slots);
        if (eff > best_eff + 0.02) {
            best_eff = eff;
            best = S;
        }
    }
    return best;
}

// Column splits for the tensor-core tiles.  Every split of a row tile starts
// its candidate lists empty, and the insertions while a list fills dominate the
// epilogue, so split only to give a small grid its first full wave: measured
// on 200k x 61, one split ran 30 ms against 42 ms for the seven that balance
// the waves best.
int choose_splits_tc(int row_tiles, int col_tiles, int slots) {
    if (row_tiles >= slots) return 1;
    return std::max(1, std::min({kMaxSplits, col_tiles, slots / std::max(row_tiles, 1)}));
}

struct KnnPlan {
    int n, m, d, dk, k, KP;
    int64_t n_pad, m_pad;
    bool alias;
    int col_tiles;
    int chunk_rows;  // multiple of kBM
    bool prune;      // carve the buffers of the pruned search (prune.cu)
};

KnnPlan make_knn_plan(int64_t n, int64_t m, int d, int k, bool alias, bool prune = true) {
    KnnPlan p{};
    p.prune = prune;
    p.n = static_cast<int>(n);
    p.m = static_cast<int>(m);
    p.d = d;
    p.dk = padded_features(d);
    p.k = k;
    p.KP = k <= 12 ? 16 : 32;
    p.n_pad = round_up(std::max<int64_t>(n, 1), kBM);
    p.m_pad = alias ? p.n_pad : round_up(m, kBN);
    p.alias = alias;
    p.col_tiles = static_cast<int>(p.m_pad / kBN);
    const int64_t per_row = static_cast<int64_t>(kMaxSplits) * p.KP * 8;
    int64_t rows = static_cast<int64_t>(kPartialBudget) / per_row / kBM * kBM;
    rows = std::max<int64_t>(rows, kBM);
    p.chunk_rows = static_cast<int>(std::min<int64_t>(rows, p.n_pad));
    return p;
}

// Spatial order of the tensor-core k-NN (order.cu): 128 pivots, used when the
// column set has at least this many points (below it the sweep is short and
// the order buys nothing).
constexpr int kSpatialPivots = 128;
constexpr int kSpatialBuckets = 64;  // distance buckets per pivot cell
constexpr int kSpatialMinCols = 16384;
static_assert(kSpatialPivots == kPrunePivots, "the pruned search bounds blocks by the order's pivots");

struct KnnBufs {
    float *Xf, *Xp, *Xlo, *xnorm, *Yf, *Yp, *Ylo, *ynorm;
    float *ynmin;  // [m_pad / 32] least column norm per batch (tensor tile)
    float *part_key;
    int *part_idx;
    SpatialOrder order;  // pointers null when not carved
    PruneBufs prune;     // pointers null when not carved
    int *fb_rows;
    DevStatus *st;
    int32_t *list_idx;  // core distances without caller lists
    float *list_dist;
};

void carve_knn(Carver &c, const KnnPlan &p, KnnBufs &b, bool own_lists) {
    b.Xf = c.take<float>(static_cast<size_t>(p.dk) * p.n_pad);
    // the tensor-core tile's low parts exist only where that engine can run
    const bool lo = p.dk <= kTensorDkMax;
    b.Xp = c.take<float>(static_cast<size_t>(p.dk) * p.n_pad);
    b.Xlo = lo ? c.take<float>(static_cast<size_t>(p.dk) * p.n_pad) : nullptr;
    b.xnorm = c.take<float>(p.n_pad);
    if (p.alias) {
        b.Yf = b.Xf;
        b.Yp = b.Xp;
        b.Ylo = b.Xlo;
        b.ynorm = b.xnorm;
    } else {
        b.Yf = c.take<float>(static_cast<size_t>(p.dk) * p.m_pad);
        b.Yp = c.take<float>(static_cast<size_t>(p.dk) * p.m_pad);
        b.Ylo = lo ? c.take<float>(static_cast<size_t>(p.dk) * p.m_pad) : nullptr;
        b.ynorm = c.take<float>(p.m_pad);
    }
    b.ynmin = lo ? c.take<float>(p.m_pad / 32) : nullptr;
    b.order = SpatialOrder{};
    b.prune = PruneBufs{};
    if (lo) {
        SpatialOrder &o = b.order;
        const int P = kSpatialPivots, NB = kSpatialPivots * kSpatialBuckets;
        o.pivots = P;
        o.buckets = kSpatialBuckets;
        o.cellY = c.take<int>(p.m_pad);
        o.permY = c.take<int>(p.m_pad);
        o.invY = c.take<int>(p.m_pad);
        o.startY = c.take<int>(NB + 1);
        o.dcellY = c.take<float>(p.m_pad);
        o.pdY = p.prune ? c.take<float>(static_cast<size_t>(p.m_pad) * P) : nullptr;
        if (p.alias) {
            o.cellX = o.cellY;
            o.permX = o.permY;
            o.invX = o.invY;
            o.startX = o.startY;
            o.dcellX = o.dcellY;
            o.pdX = o.pdY;
        } else {
            o.cellX = c.take<int>(p.n_pad);
            o.permX = c.take<int>(p.n_pad);
            o.invX = c.take<int>(p.n_pad);
            o.startX = c.take<int>(NB + 1);
            o.dcellX = c.take<float>(p.n_pad);
            o.pdX = p.prune ? c.take<float>(static_cast<size_t>(p.n_pad) * P) : nullptr;
        }
        o.counters = c.take<int>(spatial_counter_ints(P, kSpatialBuckets));
        o.tile_start = c.take<int>(p.n_pad / kBM);
        o.pivf = c.take<float>(static_cast<size_t>(kSpatialMaxD) * P);
        if (p.prune) {
            PruneBufs &q = b.prune;
            const size_t tiles = static_cast<size_t>(p.chunk_rows / kBM);
            q.Lm = c.take<float>(static_cast<size_t>(P) * p.col_tiles);
            q.Hm = c.take<float>(static_cast<size_t>(P) * p.col_tiles);
            q.HLt = c.take<float2>(static_cast<size_t>(P) * p.col_tiles);
            q.bcell = c.take<int>(p.col_tiles);
            q.minH = c.take<float>(2 * P);
            q.home_lo = c.take<int>(tiles);
            q.home = c.take<int>(tiles * kHomeBlocks);
            q.list = c.take<int>(tiles * p.col_tiles);
            q.count = c.take<int>(tiles);
            q.order = c.take<int>(tiles);
            q.slabs = c.take<int>(tiles);
            q.gthr = c.take<unsigned>(static_cast<size_t>(p.chunk_rows));
        }
    }
    const size_t part = static_cast<size_t>(kMaxSplits) * p.chunk_rows * p.KP;
    b.part_key = c.take<float>(part);
    b.part_idx = c.take<int>(part);
    b.fb_rows = c.take<int>(std::max(p.n, 1));
    b.st = c.take<DevStatus>(1);
    if (own_lists) {
        b.list_idx = c.take<int32_t>(static_cast<size_t>(std::max(p.n, 1)) * p.k);
        b.list_dist = c.take<float>(static_cast<size_t>(std::max(p.n, 1)) * p.k);
    } else {
        b.list_idx = nullptr;
        b.list_dist = nullptr;
    }
}

bool ws_ok(const void *ws, size_t have, size_t need) {
    return ws && (reinterpret_cast<uintptr_t>(ws) % 256 == 0) && have >= need;
}

hdbmst_status read_status(DevStatus *dev, DevStatus &host, cudaStream_t s) {
    CUDA_OK(cudaMemcpyAsync(&host, dev, sizeof(DevStatus), cudaMemcpyDeviceToHost, s));
    CUDA_OK(cudaStreamSynchronize(s));
    return HDBMST_OK;
}

// Pack, tile search, refine and exact fallback.  Writes out_idx / out_dist
// ([n, k]) and out_core (rank core_rank) when not NULL.
hdbmst_status run_knn(const KnnPlan &p, const KnnBufs &b, const float *X, int64_t ldx,
                      const float *Y, int64_t ldy, int32_t *out_idx, float *out_dist,
                      float *out_core, int core_rank, cudaStream_t s) {
    CUDA_OK(cudaMemsetAsync(b.st, 0, sizeof(DevStatus), s));
    const bool tensor = use_tensor(p.dk) && b.Xlo != nullptr;
    // the spatial order, and with it the pruned search, once the column set is
    // large enough for the bounds to pay for themselves
    const bool spatial = tensor && b.order.permY && p.m >= kSpatialMinCols;
    const int *permX = spatial ? b.order.permX : nullptr;
    const int *permY = spatial ? b.order.permY : nullptr;
    // tensor-core operands: TF32 low parts, or the FP16 halves (hi and lo, dk / 2
    // words per point each) in the same buffer, with one scale for X and Y
    const bool f16 = tensor && use_f16(p.dk);
    // the spatial order reads every value of X and Y: it also takes their
    // largest magnitude, the FP16 scale
    if (spatial)
        LAUNCH(K_PACK, s, launch_spatial_order(b.order, X, ldx, p.n, Y, ldy, p.m, p.alias, p.d, s,
                                               f16 ? &b.st->amax_bits : nullptr));
    const unsigned *amax = &b.st->amax_bits;
    uint32_t *Xh16 = f16 ? reinterpret_cast<uint32_t *>(b.Xlo) : nullptr;
    uint32_t *Xl16 = f16 ? Xh16 + p.n_pad * (p.dk / 2) : nullptr;
    uint32_t *Yh16 = f16 ? reinterpret_cast<uint32_t *>(b.Ylo) : nullptr;
    uint32_t *Yl16 = f16 ? Yh16 + p.m_pad * (p.dk / 2) : nullptr;
    float *xlo = tensor && !f16 ? b.Xlo : nullptr, *ylo = tensor && !f16 ? b.Ylo : nullptr;
    if (f16 && !spatial) {
        LAUNCH(K_PACK, s, launch_absmax(X, ldx, p.n, p.d, &b.st->amax_bits, s));
        if (!p.alias) LAUNCH(K_PACK, s, launch_absmax(Y, ldy, p.m, p.d, &b.st->amax_bits, s));
    }
    // the spatial order: points go to their sorted positions, read in caller
    // order.  The feature-major copy only the FP32 tile reads is written for
    // that tile alone; with the TF32 form its buffer holds the operands' high
    // parts instead (point-major, same size)
    const int *invX = spatial ? b.order.invX : nullptr, *invY = spatial ? b.order.invY : nullptr;
    float *Xf = tensor ? nullptr : b.Xf, *Yf = tensor ? nullptr : b.Yf;
    float *xhi = xlo ? b.Xf : nullptr, *yhi = ylo ? b.Yf : nullptr;
    if (p.alias) {
        LAUNCH(K_PACK, s, launch_pack(X, ldx, p.n, p.d, static_cast<int>(p.n_pad), p.dk, Xf,
                                      b.Xp, xlo, b.xnorm, &b.st->status, &b.st->nbmax_bits, s,
                                      nullptr, Xh16, Xl16, amax, &b.st->e0, invX, xhi));
    } else {
        LAUNCH(K_PACK, s, launch_pack(X, ldx, p.n, p.d, static_cast<int>(p.n_pad), p.dk, Xf,
                                      b.Xp, xlo, b.xnorm, &b.st->status, nullptr, s, nullptr, Xh16,
                                      Xl16, amax, &b.st->e0, invX, xhi));
        LAUNCH(K_PACK, s, launch_pack(Y, ldy, p.m, p.d, static_cast<int>(p.m_pad), p.dk, Yf,
                                      b.Yp, ylo, b.ynorm, &b.st->status, &b.st->nbmax_bits, s,
                                      nullptr, Yh16, Yl16, amax, &b.st->e0, invY, yhi));
    }
    // the least column norm of every 32 columns: the tensor tile's floor of
    // a batch's t
    if (tensor) LAUNCH(K_PACK, s, launch_norm_min32(b.ynorm, p.m_pad, b.ynmin, s));
    TcOperands ops{};
    if (f16)
        ops = TcOperands{Xh16, Xl16, Yh16, Yl16};
    else
        ops = TcOperands{b.Xf, b.Xlo, b.Yf, b.Ylo};
    const double tc_err = f16 ? tc::err_coef_f16(p.d, p.dk) : tc::err_coef(p.d, p.dk);
    // pruned search: the spatial order's pivots bound the column blocks (prune.cu)
    const bool prune = spatial && b.prune.list != nullptr;
    const int nh = home_blocks(p.col_tiles);
    if (prune)
        LAUNCH(K_PRUNE, s, launch_prune_setup(b.order, b.prune, p.m, p.col_tiles, p.d, s));
    const int slots = (tensor ? 1 : 2) * sm_count();
    for (int base = 0; base < p.n; base += p.chunk_rows) {
        const int rows = std::min(p.chunk_rows, p.n - base);
        const int row_tiles = (rows + kBM - 1) / kBM;
        // the second pass dispatches its row tiles longest list first when
        // they can be ordered, one CTA each; otherwise a long list is split
        // over up to kPruneChunks CTAs so that it does not finish alone
        const bool ordered = prune && row_tiles <= kOrderMax;
        const int chunks = ordered ? 1 : kPruneChunks;
        const int chunk_cap = (p.col_tiles + chunks - 1) / chunks;
        const int S0 = prune ? 1 + chunks
                     : tensor ? choose_splits_tc(row_tiles, p.col_tiles, slots)
                              : choose_splits(row_tiles, p.col_tiles, slots);
        const int tps = (p.col_tiles + S0 - 1) / S0;
        const int S = prune ? S0 : (p.col_tiles + tps - 1) / tps;
        KnnTileArgs ta{};
        ta.Xf = b.Xf;
        ta.Yf = b.Yf;
        ta.ynorm = b.ynorm;
        ta.ynmin = b.ynmin;
        ta.ldx = p.n_pad;
        ta.ldy = p.m_pad;
        ta.dk = p.dk;
        ta.row_base = base;
        ta.row_end = p.n;
        ta.chunk_rows_pad = p.chunk_rows;
        ta.col_tiles = p.col_tiles;
        ta.tiles_per_split = tps;
        ta.part_key = b.part_key;
        ta.part_idx = b.part_idx;
        ta.Xp = b.Xp;
        ta.Yp = b.Yp;
        ta.m = p.m;
        ta.status = &b.st->status;
        ta.tile_start = spatial ? b.order.tile_start : nullptr;
        ta.f16 = f16 ? 1 : 0;
        ta.amax_bits = amax;
        if (prune) {
            // home pass: slab 0, the nh blocks around the tile's own bin
            PruneHomeArgs ha{};
            ha.o = &b.order;
            ha.n = p.n;
            ha.m = p.m;
            ha.col_tiles = p.col_tiles;
            ha.row_tile0 = base / kBM;
            ha.row_tiles = row_tiles;
            ha.nh = nh;
            ha.alias = p.alias;
            LAUNCH(K_PRUNE, s, launch_prune_home(ha, b.prune, s));
            KnnTileArgs h = ta;
            h.tile_start = nullptr;
            h.blist = b.prune.home;
            h.bcount = nullptr;
            h.blist_count = nh;
            h.blist_stride = kHomeBlocks;
            h.chunk_cap = kHomeBlocks;
            h.slab_base = 0;
            LAUNCH(K_KNN_TILE, s, launch_tc_knn(p.KP, h, ops, p.n_pad, p.m_pad, row_tiles, 1, s));
            // the blocks each row tile still needs, from the home pass's bounds
            PruneListArgs pa{};
            pa.part_key = b.part_key;
            pa.part_idx = b.part_idx;
            pa.chunk_rows_pad = p.chunk_rows;
            pa.KP = p.KP;
            pa.k = p.k;
            pa.d = p.d;
            pa.xnorm = b.xnorm;
            pa.ynorm = b.ynorm;
            pa.err_c = coef_up(tc_err);
            pa.e0 = &b.st->e0;
            pa.col_tiles = p.col_tiles;
            pa.row_base = base;
            pa.row_end = p.n;
            pa.row_tiles = row_tiles;
            pa.chunk_cap = chunk_cap;
            pa.nh = nh;
            pa.blocks_total = &b.st->tile_blocks;
            pa.pdX = b.order.pdX;
            pa.permX = b.order.permX;
            LAUNCH(K_PRUNE, s, launch_prune_lists(pa, b.prune, s));
            if (ordered)
                LAUNCH(K_PRUNE, s, launch_tile_order(b.prune.count, row_tiles, b.prune.order, s));
            // second pass: slabs 1 .., in chunks of chunk_cap blocks, the
            // longest lists first
            KnnTileArgs q = ta;
            q.tile_order = ordered ? b.prune.order : nullptr;
            q.tile_start = nullptr;
            q.blist = b.prune.list;
            q.bcount = b.prune.count;
            q.blist_stride = p.col_tiles;
            q.chunk_cap = chunk_cap;
            q.slab_base = 1;
            q.seed = b.part_key;
            q.seed_idx = b.part_idx;
            q.home_lo = b.prune.home_lo;
            q.nh = nh;
            // a CTA per row tile shares its thresholds with no other CTA
            q.gthr = ordered ? nullptr : b.prune.gthr;
            LAUNCH(K_KNN_TILE, s, launch_tc_knn(p.KP, q, ops, p.n_pad, p.m_pad, row_tiles,
                                                chunks, s));
        } else if (tensor) {
            LAUNCH(K_KNN_TILE, s, launch_tc_knn(p.KP, ta, ops, p.n_pad, p.m_pad, row_tiles, S, s));
        } else {
            LAUNCH(K_KNN_TILE, s, launch_knn_tile(p.KP, ta, row_tiles, S, s));
        }
        KnnRefineArgs ra{};
        ra.part_key = b.part_key;
        ra.part_idx = b.part_idx;
        ra.splits = S;
        ra.chunk_rows_pad = p.chunk_rows;
        ra.row_base = base;
        ra.row_end = p.n;
        ra.Xp = b.Xp;
        ra.Yp = b.Yp;
        ra.xnorm = b.xnorm;
        ra.ynorm = b.ynorm;
        ra.nbmax_bits = &b.st->nbmax_bits;
        ra.err_c = coef_up(tensor ? tc_err : (2.0 * p.d + 10.0) * 0x1p-24 * 1.01);
        ra.e0 = &b.st->e0;
        ra.d = p.d;
        ra.dk = p.dk;
        ra.k = p.k;
        ra.m = p.m;
        ra.core_rank = out_core ? core_rank : 0;
        ra.out_idx = out_idx;
        ra.out_dist = out_dist;
        ra.out_core = out_core;
        ra.fb_count = &b.st->fb_count;
        ra.fb_rows = b.fb_rows;
        ra.permX = permX;
        ra.permY = permY;
        ra.tile_slabs = prune ? b.prune.slabs : nullptr;
        LAUNCH(K_KNN_REFINE, s, launch_knn_refine(p.KP, ra, rows, s));
    }
    KnnExactArgs xa{};
    xa.fb_count = &b.st->fb_count;
    xa.fb_rows = b.fb_rows;
    xa.Xp = b.Xp;
    xa.Yp = b.Yp;
    xa.dk = p.dk;
    xa.k = p.k;
    xa.m = p.m;
    xa.core_rank = out_core ? core_rank : 0;
    xa.out_idx = out_idx;
    xa.out_dist = out_dist;
    xa.out_core = out_core;
    // queued rows search their columns in up to 32 ranges of >= 4096 columns,
    // partial lists in the (now idle) candidate-list buffer
    xa.part = reinterpret_cast<unsigned long long *>(b.part_key);
    xa.permX = permX;
    xa.permY = permY;
    xa.splits = std::max(1, std::min(32, p.m / 4096));
    {
        const int64_t slots = static_cast<int64_t>(kMaxSplits) * p.chunk_rows * p.KP / 2;
        xa.rows_cap = static_cast<int>(
            std::min<int64_t>(8192, slots / (static_cast<int64_t>(xa.splits) * p.KP)));
    }
    LAUNCH(K_KNN_EXACT, s, launch_knn_exact(p.KP, xa, 2 * sm_count(), s));
    DevStatus h{};
    hdbmst_status st = read_status(b.st, h, s);
    if (st != HDBMST_OK) return st;
    g_knn_exact_rows = h.fb_count;
    g_knn_tile_pairs = prune ? static_cast<int64_t>(h.tile_blocks) * kBM * kBN
                             : static_cast<int64_t>((p.n + kBM - 1) / kBM) * p.col_tiles * kBM * kBN;
    if (h.status & kStatusNonFinite) return HDBMST_ERR_NONFINITE;
    if (h.status & kStatusTimeout) return HDBMST_ERR_TIMEOUT;
    return HDBMST_OK;
}

// ------------------------------------------------------------------ MST layout

struct MstPlan {
    int n, d, dk, L;
    int64_t n_pad;
    int index_bits;
    bool sprune;  // buffers of the pruned symmetric scan
};

MstPlan make_mst_plan(int64_t n, int d, int L) {
    MstPlan p{};
    p.n = static_cast<int>(n);
    p.d = d;
    p.dk = padded_features(d);
    p.L = L;
    p.n_pad = round_up(std::max<int64_t>(n, 1), kBM);
    int bits = 1;
    while (bits < 31 && (int64_t(1) << bits) <= std::max<int64_t>(n - 1, 1)) ++bits;
    p.index_bits = bits;
    // the pruned symmetric scan: nearest lists (bounds), the tensor-core
    // scan's feature counts, enough points, and blocks^2 arrays that stay small
    p.sprune = L > 0 && p.dk <= 64 && n >= kSymPruneMinN && p.n_pad / kBM <= kSymPruneMaxBlocks;
    return p;
}

struct MstBufs {
    float *Xf, *Xp, *Xhi, *Xlo, *Xs, *norm, *Xa, *act_core, *act_norm, *col_core, *col_norm;
    float *nmin;  // [n_pad / 32] least column norm per batch of the tensor scans
    float *Xs_hi, *Xs_lo, *Xa_hi, *Xa_lo;  // point-major grouped columns / active rows
    int *act_comp, *act_idx, *comp, *parent, *root_of, *perm, *col_comp, *start, *act_start;
    int *counters;  // [4n + 8]: size, act_size, cursor, act_cursor, totals (zeroed per round)
    unsigned char *act_flag;
    unsigned long long *part_key;
    float *part_tau;
    int *fb_rows;
    unsigned long long *cand, *ck64, *cache;
    unsigned *chi, *ub;
    unsigned char *proven;
    int *e_lo, *e_hi, *lo2, *hi2;
    unsigned *e_w, *w2, *hist;
    DevStatus *st;
    SymPruneBufs sp;  // all null unless the plan's sprune
};

void carve_mst(Carver &c, const MstPlan &p, MstBufs &b) {
    const size_t n = static_cast<size_t>(std::max(p.n, 1));
    b.Xf = c.take<float>(static_cast<size_t>(p.dk) * p.n_pad);
    b.Xp = c.take<float>(static_cast<size_t>(p.dk) * p.n_pad);
    b.norm = c.take<float>(p.n_pad);
    b.Xa = c.take<float>(static_cast<size_t>(p.dk) * p.n_pad);
    b.act_core = c.take<float>(p.n_pad);
    b.act_comp = c.take<int>(p.n_pad);
    b.act_norm = c.take<float>(p.n_pad);
    b.Xs = c.take<float>(static_cast<size_t>(p.dk) * p.n_pad);
    b.Xlo = c.take<float>(static_cast<size_t>(p.dk) * p.n_pad);
    // the TF32 form's high parts, where the tensor-core scan can run
    b.Xhi = tc_scan_supported(p.dk) ? c.take<float>(static_cast<size_t>(p.dk) * p.n_pad) : nullptr;
    b.Xs_hi = c.take<float>(static_cast<size_t>(p.dk) * p.n_pad);
    b.Xs_lo = c.take<float>(static_cast<size_t>(p.dk) * p.n_pad);
    b.Xa_hi = c.take<float>(static_cast<size_t>(p.dk) * p.n_pad);
    b.Xa_lo = c.take<float>(static_cast<size_t>(p.dk) * p.n_pad);
    // column arrays in grouped order, padded to n_pad: the tensor scan
    // prefetches them a whole tile at a time (padding entries never rank)
    b.col_core = c.take<float>(p.n_pad);
    b.col_norm = c.take<float>(p.n_pad);
    b.nmin = c.take<float>(p.n_pad / 32);
    b.perm = c.take<int>(p.n_pad);
    b.col_comp = c.take<int>(n);
    b.start = c.take<int>(n);
    b.act_start = c.take<int>(n);
    b.counters = c.take<int>(4 * n + 8);
    b.act_flag = c.take<unsigned char>(n);
    b.part_key = c.take<unsigned long long>(scan_part_entries(kMaxSplits, p.n_pad));
    b.part_tau = c.take<float>(static_cast<size_t>(kMaxSplits) * p.n_pad);
    b.fb_rows = c.take<int>(n);
    b.act_idx = c.take<int>(n);
    b.comp = c.take<int>(n);
    b.parent = c.take<int>(n);
    b.root_of = c.take<int>(n);
    b.cand = c.take<unsigned long long>(n);
    b.cache = c.take<unsigned long long>(n);
    b.ck64 = c.take<unsigned long long>(n);
    b.chi = c.take<unsigned>(n);
    b.ub = c.take<unsigned>(n);
    b.proven = c.take<unsigned char>(n);
    b.e_lo = c.take<int>(n);
    b.e_hi = c.take<int>(n);
    b.e_w = c.take<unsigned>(n);
    b.lo2 = c.take<int>(n);
    b.hi2 = c.take<int>(n);
    b.w2 = c.take<unsigned>(n);
    b.hist = c.take<unsigned>(sort_hist_entries(static_cast<int>(n)));
    b.st = c.take<DevStatus>(1);
    b.sp = SymPruneBufs{};
    if (p.sprune) {
        SymPruneBufs &q = b.sp;
        SpatialOrder &o = q.order;
        const int P = kSpatialPivots, NB = kSpatialPivots * kSpatialBuckets;
        const size_t blocks = static_cast<size_t>(p.n_pad / kBM);
        const size_t chunks = (n + kSymChunk - 1) / kSymChunk;
        o.pivots = P;
        o.buckets = kSpatialBuckets;
        o.cellY = o.cellX = c.take<int>(p.n_pad);
        o.permY = o.permX = c.take<int>(p.n_pad);
        o.invY = o.invX = c.take<int>(p.n_pad);
        o.startY = o.startX = c.take<int>(NB + 1);
        o.dcellY = o.dcellX = c.take<float>(p.n_pad);
        o.pdY = o.pdX = c.take<float>(static_cast<size_t>(p.n_pad) * P);
        o.counters = c.take<int>(spatial_counter_ints(P, kSpatialBuckets));
        o.tile_start = c.take<int>(p.n_pad / kBM);
        o.pivf = c.take<float>(static_cast<size_t>(kSpatialMaxD) * P);
        q.kcount = c.take<int>(1);
        q.cidx = c.take<int>(n);
        q.cstart = c.take<int>(kSymMaxComps);
        q.off = c.take<int>(chunks * kSymMaxComps);
        q.Lb = c.take<float>(blocks * P);
        q.Hb = c.take<float>(blocks * P);
        q.bcomp = c.take<int>(blocks);
        q.LB = c.take<float>(blocks * blocks);
        q.bth = c.take<float>(blocks);
        q.home = c.take<int>(blocks * kSymHome);
        q.hcount = c.take<int>(blocks);
        q.list = c.take<int>(blocks * blocks);
        q.lcount = c.take<int>(blocks);
        q.tile_order = c.take<int>(blocks);
        q.hkey = c.take<int>(blocks);
    }
}

bool bad_sizes(int64_t n, int d) { return n < 0 || d < 1; }

// ------------------------------------------------------------------ fixed scratch

// Scratch of hdbmst_knn_noalloc: one array per GPU, part of the device image,
// so the entry point never allocates.  Host code may not take its address
// directly (that would be a host-side stand-in); the device address is looked
// up once per device with cudaGetSymbolAddress and cached.
static __device__ __align__(256) unsigned char g_noalloc_scratch[HDBMST_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (nullptr on error).
void *noalloc_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_noalloc_ptr[dev] = p;
    }
    return g_noalloc_ptr[dev];
}

// k-NN plan whose partial lists take what the fixed scratch leaves after the
// packed copies; chunk_rows = 0 when even one 128-row chunk does not fit.
KnnPlan make_knn_plan_fixed(int64_t n, int64_t m, int d, int k, bool alias, size_t capacity) {
    KnnPlan p = make_knn_plan(n, m, d, k, alias, false);
    p.chunk_rows = kBM;
    Carver c(nullptr);
    KnnBufs b{};
    carve_knn(c, p, b, false);
    if (c.off > capacity) {
        p.chunk_rows = 0;
        return p;
    }
    const size_t per_chunk_row = static_cast<size_t>(kMaxSplits) * p.KP * 8;
    const size_t spare = capacity - c.off;
    const int64_t extra = static_cast<int64_t>(spare / per_chunk_row) / kBM * kBM;
    p.chunk_rows = static_cast<int>(std::min<int64_t>(kBM + extra, p.n_pad));
    return p;
}

// Bipartite assignment scratch: right degrees, the two sides' cluster
// masses, the right step's [m][C] counts, one moved counter per round.
struct AssignBufs {
    int *deg_r;
    unsigned long long *KR, *KL;
    unsigned *counts;
    int *moved;
    DevStatus *st;
};

void carve_assign(Carver &c, int64_t m, int C, AssignBufs &b) {
    b.deg_r = c.take<int>(static_cast<size_t>(m));
    b.KR = c.take<unsigned long long>(static_cast<size_t>(C));
    b.KL = c.take<unsigned long long>(static_cast<size_t>(C));
    b.counts = c.take<unsigned>(static_cast<size_t>(m) * static_cast<size_t>(C));
    b.moved = c.take<int>(HDBMST_ASSIGN_MAX_ROUNDS);
    b.st = c.take<DevStatus>(1);
}

// Second-moment scratch: channel means, bounds, the split operands and the
// per-split partial products.
struct MomentBufs {
    double *sum;
    float *mu_hi, *mu_lo;
    int *scale_e;
    MomentStatus *st;
    uint32_t *hi, *lo;
    float *partial;
};

void carve_moment(Carver &c, int64_t n, int C, MomentBufs &b) {
    const int64_t c_pad = round_up(C, kBM);
    const int64_t S = moment_splits(n);
    b.sum = c.take<double>(static_cast<size_t>(c_pad));
    b.mu_hi = c.take<float>(static_cast<size_t>(c_pad));
    b.mu_lo = c.take<float>(static_cast<size_t>(c_pad));
    b.scale_e = c.take<int>(static_cast<size_t>(c_pad));
    b.st = c.take<MomentStatus>(1);
    b.hi = c.take<uint32_t>(static_cast<size_t>(S * c_pad * (kMomentSplit / 2)));
    b.lo = c.take<uint32_t>(static_cast<size_t>(S * c_pad * (kMomentSplit / 2)));
    const int64_t sub = moment_subsplits(static_cast<int>(c_pad), n);
    b.partial = c.take<float>(static_cast<size_t>(S * sub * c_pad * c_pad));
}

// spikes each round's left step moved, for the last assignment call
std::vector<int64_t> g_assign_moved;

}  // namespace

// ------------------------------------------------------------------ C ABI

extern "C" {

int hdbmst_version(void) { return 100; }

const char *hdbmst_last_cuda_error(void) { return cudaGetErrorName(g_last_cuda); }

const char *hdbmst_status_string(hdbmst_status status) {
    switch (status) {
        case HDBMST_OK: return "ok";
        case HDBMST_ERR_ARG: return "invalid argument";
        case HDBMST_ERR_UNSUPPORTED: return "unsupported size (k, min_samples, d or n beyond the build's limits)";
        case HDBMST_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case HDBMST_ERR_NONFINITE: return "non-finite value in the points or core distances";
        case HDBMST_ERR_NOCONVERGE: return "Boruvka made no progress";
        case HDBMST_ERR_CUDA: return "CUDA error";
        case HDBMST_ERR_TOO_LARGE: return "problem too large for the fixed scratch of hdbmst_knn_noalloc";
        case HDBMST_ERR_TIMEOUT: return "a wait inside a kernel gave up after its bound";
    }
    return "unknown status";
}

size_t hdbmst_workspace_bytes(int op, int64_t n, int64_t m, int d, int k) {
    if (op == HDBMST_OP_MOMENT) {
        if (n < 1 || n > HDBMST_MOMENT_NMAX || d < 1 || d > HDBMST_DMAX) return 0;
        Carver c(nullptr);
        MomentBufs b{};
        carve_moment(c, n, d, b);
        return c.off;
    }
    if (op == HDBMST_OP_ASSIGN) {
        if (n < 0 || n > HDBMST_ASSIGN_NMAX || m < 1 || m > HDBMST_NMAX || d < 1 ||
            d > HDBMST_ASSIGN_CMAX || k < 1 || k > HDBMST_KMAX)
            return 0;
        Carver c(nullptr);
        AssignBufs b{};
        carve_assign(c, m, d, b);
        return c.off;
    }
    if (d < 1 || d > HDBMST_DMAX || n < 0 || n > HDBMST_NMAX) return 0;
    Carver c(nullptr);
    if (op == HDBMST_OP_KNN) {
        if (m < 1 || m > HDBMST_NMAX || k < 1 || k > HDBMST_KMAX) return 0;
        KnnPlan p = make_knn_plan(n, m, d, k, false);
        KnnBufs b{};
        carve_knn(c, p, b, false);
        return c.off;
    }
    if (op == HDBMST_OP_CORE) {
        if (n < 1 || k < 1 || k > n || k + 1 > HDBMST_KMAX) return 0;
        const int L = static_cast<int>(std::min<int64_t>(k + 1, n));
        KnnPlan p = make_knn_plan(n, n, d, L, true);
        KnnBufs b{};
        carve_knn(c, p, b, true);
        return c.off;
    }
    if (op == HDBMST_OP_MST) {
        if (k < 0 || k > HDBMST_KMAX) return 0;
        MstPlan p = make_mst_plan(n, d, k);
        MstBufs b{};
        carve_mst(c, p, b);
        return c.off;
    }
    return 0;
}

hdbmst_status hdbmst_knn(const float *X, int64_t ldx, int64_t n, const float *Y, int64_t ldy,
                         int64_t m, int d, int k, int32_t *out_idx, float *out_dist,
                         void *workspace, size_t workspace_bytes, hdbmst_stream stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (bad_sizes(n, d) || m < 1 || k < 1 || k > m || ldx < n || ldy < m) return HDBMST_ERR_ARG;
    if (k > HDBMST_KMAX || d > HDBMST_DMAX || n > HDBMST_NMAX || m > HDBMST_NMAX)
        return HDBMST_ERR_UNSUPPORTED;
    if (n == 0) return HDBMST_OK;
    if (!X || !Y || !out_idx || !out_dist) return HDBMST_ERR_ARG;
    const size_t need = hdbmst_workspace_bytes(HDBMST_OP_KNN, n, m, d, k);
    if (!ws_ok(workspace, workspace_bytes, need)) return HDBMST_ERR_WORKSPACE;
    const bool alias = (X == Y && ldx == ldy && n == m);
    KnnPlan p = make_knn_plan(n, m, d, k, alias);
    Carver c(workspace);
    KnnBufs b{};
    carve_knn(c, p, b, false);
    return run_knn(p, b, X, ldx, Y, ldy, out_idx, out_dist, nullptr, 0, s);
}

hdbmst_status hdbmst_core_distances(const float *X, int64_t ldx, int64_t n, int d,
                                    int min_samples, float *out_core, int32_t *out_knn_idx,
                                    float *out_knn_dist, void *workspace,
                                    size_t workspace_bytes, hdbmst_stream stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (bad_sizes(n, d) || n < 1 || ldx < n || min_samples < 1 || min_samples > n)
        return HDBMST_ERR_ARG;
    if ((out_knn_idx == nullptr) != (out_knn_dist == nullptr)) return HDBMST_ERR_ARG;
    if (min_samples + 1 > HDBMST_KMAX || d > HDBMST_DMAX || n > HDBMST_NMAX)
        return HDBMST_ERR_UNSUPPORTED;
    if (!X || !out_core) return HDBMST_ERR_ARG;
    const size_t need = hdbmst_workspace_bytes(HDBMST_OP_CORE, n, 0, d, min_samples);
    if (!ws_ok(workspace, workspace_bytes, need)) return HDBMST_ERR_WORKSPACE;
    const int L = static_cast<int>(std::min<int64_t>(min_samples + 1, n));
    KnnPlan p = make_knn_plan(n, n, d, L, true);
    Carver c(workspace);
    KnnBufs b{};
    carve_knn(c, p, b, true);
    int32_t *li = out_knn_idx ? out_knn_idx : b.list_idx;
    float *ld = out_knn_dist ? out_knn_dist : b.list_dist;
    return run_knn(p, b, X, ldx, X, ldx, li, ld, out_core, min_samples, s);
}

hdbmst_status hdbmst_mr_mst(const float *X, int64_t ldx, int64_t n, int d, const float *core,
                            const int32_t *knn_idx, const float *knn_dist, int knn_len,
                            int32_t *out_edges, float *out_w, void *workspace,
                            size_t workspace_bytes, hdbmst_stream stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (bad_sizes(n, d) || ldx < n) return HDBMST_ERR_ARG;
    if ((knn_idx == nullptr) != (knn_dist == nullptr)) return HDBMST_ERR_ARG;
    const bool shortcuts = knn_idx != nullptr;
    if (shortcuts && (knn_len < 1 || knn_len > n)) return HDBMST_ERR_ARG;
    if (d > HDBMST_DMAX || n > HDBMST_NMAX || (shortcuts && knn_len > HDBMST_KMAX))
        return HDBMST_ERR_UNSUPPORTED;
    if (n <= 1) return HDBMST_OK;
    if (!X || !core || !out_edges || !out_w) return HDBMST_ERR_ARG;
    const int L = shortcuts ? knn_len : 0;
    const size_t need = hdbmst_workspace_bytes(HDBMST_OP_MST, n, 0, d, L);
    if (!ws_ok(workspace, workspace_bytes, need)) return HDBMST_ERR_WORKSPACE;

    MstPlan p = make_mst_plan(n, d, L);
    Carver c(workspace);
    MstBufs b{};
    carve_mst(c, p, b);
    const int N = p.n;
    const int slots = 2 * sm_count();
    const int col_tiles = static_cast<int>(p.n_pad / kBN);

    const bool tensor = use_tensor_scan(p.dk);
    // tensor-core operands: TF32 low parts, or the FP16 halves (hi and lo,
    // dk / 2 words per point each) in the same buffer
    const bool f16 = tensor && use_f16(p.dk);
    const int dkw = f16 ? p.dk / 2 : p.dk;  // 32-bit words per point of each part
    const float *op_hi = f16 ? b.Xlo : b.Xhi;
    const float *op_lo = f16 ? b.Xlo + p.n_pad * dkw : b.Xlo;
    CUDA_OK(cudaMemsetAsync(b.st, 0, sizeof(DevStatus), s));
    if (f16) LAUNCH(K_PACK, s, launch_absmax(X, ldx, N, d, &b.st->amax_bits, s));
    LAUNCH(K_PACK, s, launch_pack(X, ldx, N, d, static_cast<int>(p.n_pad), p.dk, b.Xf, b.Xp,
                                  tensor && !f16 ? b.Xlo : nullptr, b.norm, &b.st->status,
                                  &b.st->nbmax_bits, s, nullptr,
                                  f16 ? reinterpret_cast<uint32_t *>(b.Xlo) : nullptr,
                                  f16 ? reinterpret_cast<uint32_t *>(b.Xlo) + p.n_pad * dkw
                                      : nullptr,
                                  &b.st->amax_bits, &b.st->e0, nullptr,
                                  tensor && !f16 ? b.Xhi : nullptr));
    LAUNCH(K_CHECK_CORE, s, launch_check_core(core, N, &b.st->status, s));
    LAUNCH(K_MST_INIT, s, launch_mst_init(N, b.comp, b.cand, b.ck64, b.chi, b.ub, b.cache, s));

    int max_rounds = 2;
    while ((int64_t(1) << (max_rounds - 2)) < N) ++max_rounds;  // ceil(log2 n) + 2
    if (g_test_max_rounds > 0) max_rounds = std::min(max_rounds, g_test_max_rounds);
    int edges = 0;
    DevStatus h{};
    g_round_active.clear();
    g_round_edges.clear();
    g_round_exact.clear();
    g_mst_scan_pairs = 0;
    int *size = b.counters, *act_size = b.counters + N, *cursor = b.counters + 2 * N,
        *act_cursor = b.counters + 3 * N, *totals = b.counters + 4 * N;
    const float err_c = coef_up(f16      ? tc::err_coef_f16(d, p.dk)
                                : tensor ? tc::err_coef(d, p.dk)
                                         : (2.0 * d + 10.0) * 0x1p-24 * 1.01);
    g_round_sym.clear();
    // the spatial order of all points (pivots, bins, pivot distances) for the
    // pruned symmetric scan, once per call
    const bool sp_ready = p.sprune && tensor && shortcuts && g_scan_form != HDBMST_SCAN_ONE_SIDED &&
                          g_sym_prune;
    // It is first needed by round 3 or so: it runs on a side stream beside
    // the first rounds, whose one-sided scans leave most SMs idle.
    JoinOnExit sp_join{s};
    if (sp_ready) {
        SideStream *ss = nullptr;
        CUDA_OK(side_stream(&ss));
        CUDA_OK(cudaEventRecord(ss->fork, s));
        CUDA_OK(cudaStreamWaitEvent(ss->s, ss->fork, 0));
        LAUNCH(K_SYM_PRUNE, ss->s,
               launch_spatial_order(b.sp.order, X, ldx, N, X, ldx, N, true, d, ss->s));
        CUDA_OK(cudaEventRecord(ss->join, ss->s));
        sp_join.e = ss->join;
    }
    for (int round = 0; round < max_rounds && edges < N - 1; ++round) {
        int fallback = 0;
        int64_t recorded = -1;
        if (shortcuts) {
            LAUNCH(K_NBR_CANDIDATE, s, launch_nbr_candidate(N, L, knn_idx, knn_dist, core, b.comp,
                                                            b.cache, b.cand, b.proven, b.ub,
                                                            &b.st->status, s));
        }
        // the points that need a scan (act_flag) and the per-label counts
        const auto classify = [&]() -> hdbmst_status {
            CUDA_OK(cudaMemsetAsync(b.counters, 0, sizeof(int) * (4 * static_cast<size_t>(N) + 8), s));
            CUDA_OK(cudaMemsetAsync(&b.st->act_count, 0, sizeof(int), s));
            LAUNCH(K_ACTIVE, s, launch_classify(N, shortcuts ? b.proven : nullptr, core, b.comp,
                                                shortcuts ? b.ub : nullptr, b.act_flag, size,
                                                act_size, &b.st->act_count, s));
            return HDBMST_OK;
        };
        hdbmst_status rs = classify();
        if (rs != HDBMST_OK) return rs;
        rs = read_status(b.st, h, s);
        if (rs != HDBMST_OK) return rs;
        if (h.status & kStatusNonFinite) return HDBMST_ERR_NONFINITE;
        if (h.status & kStatusBadList) return HDBMST_ERR_ARG;
        int na = h.act_count;
        bool sym_done = false;
        const bool sym = na > 0 && tensor && shortcuts && g_scan_form != HDBMST_SCAN_ONE_SIDED &&
                         (g_scan_form == HDBMST_SCAN_SYMMETRIC || 2 * static_cast<int64_t>(na) >= N);
        if (sym) {
            // the set P in grouped order: rows and columns of the symmetric scan
            CUDA_OK(cudaMemsetAsync(b.counters, 0, sizeof(int) * (4 * static_cast<size_t>(N) + 8), s));
            CUDA_OK(cudaMemsetAsync(&b.st->act_count, 0, sizeof(int), s));
            CUDA_OK(cudaMemsetAsync(&b.st->sym_umax, 0, 3 * sizeof(unsigned), s));
            LAUNCH(K_ACTIVE, s, launch_sym_classify(N, b.comp, b.ub, core, &b.st->sym_umax,
                                                    b.act_flag, size, act_size, &b.st->act_count,
                                                    &b.st->sym_ncomp, s));
            rs = read_status(b.st, h, s);
            if (rs != HDBMST_OK) return rs;
            const int np = h.act_count;
            // pruned by blocks when the spatial order exists and the
            // components fit the grouping
            const bool pruned = sp_ready && h.sym_ncomp <= kSymMaxComps;
            const int np_pad = static_cast<int>(round_up(std::max(np, 1), kBM));
            LAUNCH(K_GATHER, s, launch_group(N, static_cast<int>(p.n_pad), b.comp, core, b.norm,
                                             b.act_flag, size, act_size, b.start, b.act_start,
                                             cursor, act_cursor, totals, b.perm, b.col_comp,
                                             b.col_core, b.col_norm, b.act_idx, s));
            if (pruned) {
                CUDA_OK(cudaStreamWaitEvent(s, sp_join.e, 0));  // the spatial order
                LAUNCH(K_SYM_PRUNE, s, launch_sym_group(b.sp, N, b.act_flag, b.comp, b.act_start,
                                                        act_size, b.act_idx, s));
            }
            LAUNCH(K_GATHER, s, launch_gather(np, np_pad, p.dk, b.act_idx, b.Xf, p.n_pad, core,
                                              b.comp, b.norm, nullptr, b.act_core, b.act_comp,
                                              b.act_norm, s));
            LAUNCH(K_GATHER, s, launch_gather_points(np, np_pad, dkw, b.act_idx, op_hi, op_lo,
                                                     b.Xa_hi, b.Xa_lo, s));
            // scratch of the one-sided scan, idle in this round: the tile
            // records, the bounds (the sort's buffer, used after the rounds)
            // and the list of recorded pairs
            int4 *tile_meta = reinterpret_cast<int4 *>(b.part_tau);
            unsigned *theta = b.w2;
            int2 *pairs = reinterpret_cast<int2 *>(b.part_key);
            LAUNCH(K_GATHER, s, launch_sym_prepare(N, np, np_pad, b.act_comp, b.ub, theta,
                                                   b.act_norm, tile_meta, s));
            LAUNCH(K_GATHER, s, launch_norm_min32(b.act_norm, np_pad, b.nmin, s));
            SymArgs ya{};
            ya.np = np;
            ya.ld = np_pad;
            ya.blocks = np_pad / kBM;
            ya.idx = b.act_idx;
            ya.core = b.act_core;
            ya.comp = b.act_comp;
            ya.norm = b.act_norm;
            ya.nmin = b.nmin;
            ya.comp_start = b.act_start;
            ya.comp_size = act_size;
            ya.tile_meta = tile_meta;
            ya.theta = theta;
            ya.cand = b.cand;
            ya.pairs = pairs;
            ya.pair_count = &b.st->sym_pairs;
            ya.pair_cap = list_cap(scan_part_entries(kMaxSplits, p.n_pad));
            ya.d = d;
            ya.dk = p.dk;
            ya.err_c = err_c;
            ya.e0 = &b.st->e0;
            ya.f16 = f16 ? 1 : 0;
            ya.amax_bits = &b.st->amax_bits;
            ya.tile_pairs = &b.st->scan_pairs;
            ya.status = &b.st->status;
            if (pruned) {
                // bounds of the blocks, the home pass, then the lists
                const int blocks = np_pad / kBM;
                LAUNCH(K_SYM_PRUNE, s, launch_sym_blocks(b.sp, np, blocks, b.act_idx, b.act_comp, d, s));
                SymArgs ha = ya;
                ha.list = b.sp.home;
                ha.list_count = b.sp.hcount;
                ha.list_stride = kSymHome;
                if (blocks <= kOrderMax) {
                    // the row tiles nearest another component (the most work) first
                    LAUNCH(K_SYM_PRUNE, s,
                           launch_tile_order(b.sp.hkey, blocks, b.sp.tile_order, s));
                    ha.tile_order = b.sp.tile_order;
                }
                LAUNCH(K_SCAN, s, launch_tc_sym(ha, b.Xa_hi, b.Xa_lo, s));
                LAUNCH(K_SYM_PRUNE, s, launch_sym_lists(b.sp, np, blocks, b.act_comp, theta, d, s));
                ya.list = b.sp.list;
                ya.list_count = b.sp.lcount;
                ya.list_stride = blocks;
                if (blocks <= kOrderMax) {
                    // the longest lists first
                    LAUNCH(K_SYM_PRUNE, s,
                           launch_tile_order(b.sp.lcount, blocks, b.sp.tile_order, s));
                    ya.tile_order = b.sp.tile_order;
                }
            }
            LAUNCH(K_SCAN, s, launch_tc_sym(ya, b.Xa_hi, b.Xa_lo, s));
            rs = read_status(b.st, h, s);
            if (rs != HDBMST_OK) return rs;
            if (h.status & kStatusTimeout) return HDBMST_ERR_TIMEOUT;
            if (h.sym_pairs <= ya.pair_cap) {
                LAUNCH(K_SCAN_REFINE, s, launch_sym_pairs_exact(pairs, h.sym_pairs, b.act_idx, b.Xp,
                                                                p.dk, core, b.cand, s));
                sym_done = true;
                recorded = h.sym_pairs;
                na = np;
            } else {
                // the list overflowed: this round one-sided
                rs = classify();
                if (rs != HDBMST_OK) return rs;
                rs = read_status(b.st, h, s);
                if (rs != HDBMST_OK) return rs;
                na = h.act_count;
            }
        }
        if (na > 0 && !sym_done) {
            const int na_pad = static_cast<int>(round_up(na, kBM));
            LAUNCH(K_GATHER, s, launch_group(N, static_cast<int>(p.n_pad), b.comp, core, b.norm,
                                             b.act_flag, size, act_size, b.start, b.act_start,
                                             cursor, act_cursor, totals, b.perm, b.col_comp,
                                             b.col_core, b.col_norm, b.act_idx, s));
            LAUNCH(K_GATHER, s, launch_gather(na, na_pad, p.dk, b.act_idx, b.Xf, p.n_pad, core,
                                              b.comp, b.norm, tensor ? nullptr : b.Xa, b.act_core,
                                              b.act_comp, b.act_norm, s));
            if (tensor) {
                LAUNCH(K_GATHER, s, launch_gather_points(N, static_cast<int>(p.n_pad), dkw, b.perm,
                                                         op_hi, op_lo, b.Xs_hi, b.Xs_lo, s));
                LAUNCH(K_GATHER, s, launch_norm_min32(b.col_norm, p.n_pad, b.nmin, s));
                LAUNCH(K_GATHER, s, launch_gather_points(na, na_pad, dkw, b.act_idx, op_hi, op_lo,
                                                         b.Xa_hi, b.Xa_lo, s));
            } else {
                LAUNCH(K_GATHER, s, launch_gather_cols(N, static_cast<int>(p.n_pad), p.dk, b.perm,
                                                       b.Xf, b.Xs, s));
            }
            ScanArgs sa{};
            sa.Xa = b.Xa;
            sa.lda = na_pad;
            sa.act_idx = b.act_idx;
            sa.act_core = b.act_core;
            sa.act_comp = b.act_comp;
            sa.act_norm = b.act_norm;
            sa.na = na;
            sa.Xs = b.Xs;
            sa.ldx = p.n_pad;
            sa.col_orig = b.perm;
            sa.col_norm = b.col_norm;
            sa.col_nmin = b.nmin;
            sa.col_core = b.col_core;
            sa.col_comp = b.col_comp;
            sa.comp_start = b.start;
            sa.comp_size = size;
            sa.Xp = b.Xp;
            sa.core = core;
            sa.comp = b.comp;
            sa.nbmax_bits = &b.st->nbmax_bits;
            sa.n = N;
            sa.d = d;
            sa.dk = p.dk;
            sa.col_tiles = col_tiles;
            const int row_tiles = (na + kBM - 1) / kBM;
            // the tensor scan splits the columns so that a few active rows
            // still give every SM a CTA, as far as the partial lists' scratch
            // (kMaxSplits x n_pad rows) holds that many splits of na_pad rows
            const int scan_cap = static_cast<int>(std::min<int64_t>(
                kScanMaxSplits, static_cast<int64_t>(kMaxSplits) * p.n_pad / na_pad));
            const int S0 = tensor ? std::max(1, std::min({scan_cap, col_tiles,
                                                          (slots / 2) / std::max(row_tiles, 1)}))
                                  : choose_splits(row_tiles, col_tiles, slots);
            const int tps = (col_tiles + S0 - 1) / S0;
            const int S = (col_tiles + tps - 1) / tps;
            sa.tiles_per_split = tps;
            sa.splits = S;
            sa.part_key = b.part_key;
            sa.part_tau = b.part_tau;
            sa.cand = b.cand;
            sa.fb_count = &b.st->fb_count;
            sa.fb_rows = b.fb_rows;
            sa.status = &b.st->status;
            sa.err_c = err_c;
            sa.e0 = &b.st->e0;
            sa.f16 = f16 ? 1 : 0;
            sa.amax_bits = &b.st->amax_bits;
            sa.tile_pairs = &b.st->scan_pairs;
            // the component bounds: a threshold per row (tensor scan) and the
            // refine's acceptance of rows with no edge at or below U_C
            sa.ub = tensor && shortcuts ? b.ub : nullptr;
            sa.act_flag = b.act_flag;
            CUDA_OK(cudaMemsetAsync(&b.st->fb_count, 0, sizeof(int), s));
            if (tensor) {
                LAUNCH(K_SCAN, s, launch_tc_scan(sa, b.Xa_hi, b.Xa_lo, b.Xs_hi, b.Xs_lo, row_tiles,
                                                 S, s));
            } else {
                LAUNCH(K_SCAN, s, launch_scan(sa, row_tiles, S, s));
            }
            LAUNCH(K_SCAN_REFINE, s, launch_scan_refine(sa, s));
            rs = read_status(b.st, h, s);
            if (rs != HDBMST_OK) return rs;
            if (h.status & kStatusTimeout) return HDBMST_ERR_TIMEOUT;
            const int nf = h.fb_count;
            fallback = nf;
            bool rescanned = false;
            if (nf > 0 && tensor) {
                // rows the rounding proof left open, on the tensor cores: each
                // row's key drops to its exact cheapest edge (tc_sym.cu)
                const int nf_pad = static_cast<int>(round_up(nf, kBM));
                LAUNCH(K_GATHER, s, launch_gather(nf, nf_pad, p.dk, b.fb_rows, b.Xf, p.n_pad,
                                                  core, b.comp, b.norm, nullptr, b.act_core,
                                                  b.act_comp, b.act_norm, s));
                LAUNCH(K_GATHER, s, launch_gather_points(nf, nf_pad, dkw, b.fb_rows, op_hi, op_lo,
                                                         b.Xa_hi, b.Xa_lo, s));
                CUDA_OK(cudaMemsetAsync(&b.st->sym_pairs, 0, sizeof(int), s));
                RescanArgs ra{};
                ra.nr = nf;
                ra.row_idx = b.fb_rows;
                ra.row_norm = b.act_norm;
                ra.row_core = b.act_core;
                ra.row_comp = b.act_comp;
                ra.n = N;
                ra.ldx = p.n_pad;
                ra.col_norm = b.col_norm;
                ra.col_core = b.col_core;
                ra.col_orig = b.perm;
                ra.comp_start = b.start;
                ra.comp_size = size;
                ra.col_tiles = col_tiles;
                const int xt = (nf + kBM - 1) / kBM;
                const int X0 = std::max(1, std::min(col_tiles, sm_count() / xt));
                ra.tiles_per_split = (col_tiles + X0 - 1) / X0;
                const int xs = (col_tiles + ra.tiles_per_split - 1) / ra.tiles_per_split;
                ra.cand = b.cand;
                // the scan's candidate slabs, read by the refine before this
                int2 *pairs = reinterpret_cast<int2 *>(b.part_key);
                ra.pairs = pairs;
                ra.pair_count = &b.st->sym_pairs;
                ra.pair_cap = list_cap(scan_part_entries(kMaxSplits, p.n_pad));
                ra.d = d;
                ra.dk = p.dk;
                ra.err_c = err_c;
                ra.e0 = &b.st->e0;
                ra.f16 = f16 ? 1 : 0;
                ra.amax_bits = &b.st->amax_bits;
                ra.status = &b.st->status;
                LAUNCH(K_SCAN_EXACT, s, launch_tc_rescan(ra, b.Xa_hi, b.Xa_lo, b.Xs_hi, b.Xs_lo,
                                                         xt, xs, s));
                rs = read_status(b.st, h, s);
                if (rs != HDBMST_OK) return rs;
                if (h.status & kStatusTimeout) return HDBMST_ERR_TIMEOUT;
                if (h.sym_pairs <= ra.pair_cap) {
                    LAUNCH(K_SCAN_EXACT, s, launch_sym_pairs_exact(pairs, h.sym_pairs, nullptr,
                                                                   b.Xp, p.dk, core, b.cand, s));
                    rescanned = true;
                }
            }
            if (nf > 0 && !rescanned) {
                // rows the rounding proof left open: gather them as rows and
                // search them again with the exact weight
                if (tensor)
                    LAUNCH(K_GATHER, s, launch_gather_cols(N, static_cast<int>(p.n_pad), p.dk,
                                                           b.perm, b.Xf, b.Xs, s));
                const int nf_pad = static_cast<int>(round_up(nf, kBM));
                LAUNCH(K_GATHER, s, launch_gather(nf, nf_pad, p.dk, b.fb_rows, b.Xf, p.n_pad,
                                                  core, b.comp, b.norm, b.Xa, b.act_core,
                                                  b.act_comp, b.act_norm, s));
                ScanArgs xa = sa;
                xa.tile_pairs = nullptr;  // the exact re-scan is not the ranking tile
                xa.ub = nullptr;
                xa.lda = nf_pad;
                xa.act_idx = b.fb_rows;
                xa.na = nf;
                const int xt = (nf + kBM - 1) / kBM;
                // no partial lists here (atomicMin per row), so split the
                // columns finely enough to give every CTA slot work
                const int X0 = std::max(1, std::min(col_tiles, (slots + xt - 1) / xt));
                const int xtps = (col_tiles + X0 - 1) / X0;
                xa.tiles_per_split = xtps;
                xa.splits = (col_tiles + xtps - 1) / xtps;
                LAUNCH(K_SCAN_EXACT, s, launch_scan_exact(xa, xt, xa.splits, s));
            }
        }
        LAUNCH(K_COMP_MIN, s, launch_comp_min(N, b.cand, b.comp, b.ck64, b.chi, b.proven,
                                              sym_done ? nullptr : b.act_flag,
                                              shortcuts ? b.cache : nullptr, s, 0));
        LAUNCH(K_COMP_MIN, s, launch_comp_min(N, b.cand, b.comp, b.ck64, b.chi, nullptr, nullptr,
                                              nullptr, s, 1));
        LAUNCH(K_HOOK, s, launch_hook(N, b.comp, b.ck64, b.chi, b.parent, b.e_lo, b.e_hi,
                                      reinterpret_cast<float *>(b.e_w), &b.st->edge_count,
                                      &b.st->status, s));
        LAUNCH(K_ROOTS, s, launch_roots(N, N - edges, b.comp, b.parent, b.root_of,
                                        b.st->jump_live, round + 1, sm_count(), s,
                                        g_test_jump_launches));
        LAUNCH(K_RELABEL, s, launch_relabel(N, b.comp, b.root_of, b.parent, b.cand, b.ck64, b.chi,
                                            b.ub, &b.st->status, s));
        rs = read_status(b.st, h, s);
        if (rs != HDBMST_OK) return rs;
        if (h.status & kStatusNonFinite) return HDBMST_ERR_NONFINITE;
        if (h.status & (kStatusNoConverge | kStatusOverflow)) return HDBMST_ERR_NOCONVERGE;
        if (h.edge_count <= edges) return HDBMST_ERR_NOCONVERGE;
        edges = h.edge_count;
        g_round_active.push_back(na);
        g_round_edges.push_back(edges);
        g_round_exact.push_back(fallback);
        g_round_sym.push_back(recorded);
    }
    g_mst_scan_pairs = static_cast<int64_t>(h.scan_pairs);
    if (edges != N - 1) return HDBMST_ERR_NOCONVERGE;
    cudaError_t e = sort_edges(N - 1, p.index_bits, b.e_w, b.e_lo, b.e_hi, b.w2, b.lo2, b.hi2,
                               b.hist, out_edges, out_w, s, before, after);
    return e == cudaSuccess ? HDBMST_OK : cuda_fail(e);
}

hdbmst_status hdbmst_knn_noalloc(const float *X, int64_t ldx, int64_t n, const float *Y,
                                 int64_t ldy, int64_t m, int d, int k, int32_t *out_idx,
                                 float *out_dist, hdbmst_stream stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (bad_sizes(n, d) || m < 1 || k < 1 || k > m || ldx < n || ldy < m) return HDBMST_ERR_ARG;
    if (k > HDBMST_KMAX || d > HDBMST_DMAX || n > HDBMST_NMAX || m > HDBMST_NMAX)
        return HDBMST_ERR_UNSUPPORTED;
    if (n == 0) return HDBMST_OK;
    if (!X || !Y || !out_idx || !out_dist) return HDBMST_ERR_ARG;
    const bool alias = (X == Y && ldx == ldy && n == m);
    KnnPlan p = make_knn_plan_fixed(n, m, d, k, alias, HDBMST_NOALLOC_SCRATCH_BYTES);
    if (p.chunk_rows == 0) return HDBMST_ERR_TOO_LARGE;
    Carver need(nullptr);
    KnnBufs nb{};
    carve_knn(need, p, nb, false);
    if (need.off > HDBMST_NOALLOC_SCRATCH_BYTES) return HDBMST_ERR_TOO_LARGE;
    void *scratch = noalloc_scratch();
    if (!scratch) return HDBMST_ERR_CUDA;
    Carver c(scratch);
    KnnBufs b{};
    carve_knn(c, p, b, false);
    return run_knn(p, b, X, ldx, Y, ldy, out_idx, out_dist, nullptr, 0, s);
}

hdbmst_status hdbmst_bipartite_assign(const int32_t *nbr, int64_t n, int k, int64_t m,
                                      int n_clusters, double gamma, const int32_t *right_init,
                                      int32_t *out_left, int32_t *out_right, int max_rounds,
                                      int *out_rounds, void *workspace, size_t workspace_bytes,
                                      hdbmst_stream stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    g_assign_moved.clear();
    if (n < 0 || m < 1 || k < 1 || n_clusters < 1 || max_rounds < 1 || !(gamma >= 0.0) ||
        !std::isfinite(gamma))
        return HDBMST_ERR_ARG;
    if (k > HDBMST_KMAX || n > HDBMST_ASSIGN_NMAX || m > HDBMST_NMAX ||
        n_clusters > HDBMST_ASSIGN_CMAX || max_rounds > HDBMST_ASSIGN_MAX_ROUNDS)
        return HDBMST_ERR_UNSUPPORTED;
    if (!right_init || !out_right || (n > 0 && (!nbr || !out_left))) return HDBMST_ERR_ARG;
    const size_t need = hdbmst_workspace_bytes(HDBMST_OP_ASSIGN, n, m, n_clusters, k);
    if (!ws_ok(workspace, workspace_bytes, need)) return HDBMST_ERR_WORKSPACE;
    Carver c(workspace);
    AssignBufs b{};
    carve_assign(c, m, n_clusters, b);
    const int N = static_cast<int>(n), M = static_cast<int>(m), C = n_clusters;
    CUDA_OK(cudaMemsetAsync(b.st, 0, sizeof(DevStatus), s));
    CUDA_OK(cudaMemsetAsync(b.deg_r, 0, sizeof(int) * static_cast<size_t>(M), s));
    CUDA_OK(cudaMemsetAsync(b.moved, 0, sizeof(int) * HDBMST_ASSIGN_MAX_ROUNDS, s));
    if (out_right != right_init)
        CUDA_OK(cudaMemcpyAsync(out_right, right_init, sizeof(int32_t) * static_cast<size_t>(M),
                                cudaMemcpyDeviceToDevice, s));
    // indices and initial labels are checked before any kernel uses them
    LAUNCH(K_ASSIGN_INIT, s, launch_assign_degree(nbr, N, k, M, b.deg_r, out_left, &b.st->status, s));
    LAUNCH(K_ASSIGN_INIT, s, launch_assign_right_mass(out_right, M, C, b.deg_r, b.KR,
                                                      &b.st->status, s));
    DevStatus h{};
    hdbmst_status rs = read_status(b.st, h, s);
    if (rs != HDBMST_OK) return rs;
    if (h.status & kStatusBadList) return HDBMST_ERR_ARG;
    int rounds = 0;
    for (int round = 0; round < max_rounds; ++round) {
        if (round > 0)
            LAUNCH(K_ASSIGN_LEFT, s, launch_assign_right_mass(out_right, M, C, b.deg_r, b.KR,
                                                              &b.st->status, s));
        LAUNCH(K_ASSIGN_LEFT, s, launch_assign_left(nbr, N, k, C, out_right, b.KR, gamma, out_left,
                                                    b.KL, b.moved + round, s));
        int moved = 0;
        CUDA_OK(cudaMemcpyAsync(&moved, b.moved + round, sizeof(int), cudaMemcpyDeviceToHost, s));
        CUDA_OK(cudaStreamSynchronize(s));
        ++rounds;
        g_assign_moved.push_back(moved);
        if (moved == 0) break;
        LAUNCH(K_ASSIGN_RIGHT, s, launch_assign_right(nbr, N, k, M, C, out_left, b.deg_r, b.KL,
                                                      gamma, b.counts, out_right, s));
    }
    if (out_rounds) *out_rounds = rounds;
    return HDBMST_OK;
}

hdbmst_status hdbmst_second_moment(const float *X, int64_t ld, int channels, int64_t t0,
                                   int64_t n, int centred, int accumulate, float *out,
                                   void *workspace, size_t workspace_bytes,
                                   hdbmst_stream stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (channels < 1 || n < 1 || t0 < 0 || ld < t0 + n || !X || !out) return HDBMST_ERR_ARG;
    if (channels > HDBMST_DMAX || n > HDBMST_MOMENT_NMAX) return HDBMST_ERR_UNSUPPORTED;
    if (!moment_supported()) return HDBMST_ERR_UNSUPPORTED;
    const size_t need = hdbmst_workspace_bytes(HDBMST_OP_MOMENT, n, 0, channels, 0);
    if (!ws_ok(workspace, workspace_bytes, need)) return HDBMST_ERR_WORKSPACE;
    Carver c(workspace);
    MomentBufs b{};
    carve_moment(c, n, channels, b);
    const int c_pad = static_cast<int>(round_up(channels, kBM));
    const int cen = centred ? 1 : 0;
    CUDA_OK(cudaMemsetAsync(b.st, 0, sizeof(MomentStatus), s));
    CUDA_OK(cudaMemsetAsync(b.scale_e, 0, sizeof(int) * static_cast<size_t>(c_pad), s));
    LAUNCH(K_MOMENT_PREP, s, launch_moment_stats(X, ld, channels, t0, n, b.sum, b.mu_hi, b.mu_lo,
                                                 b.scale_e, b.st, s));
    LAUNCH(K_MOMENT_PREP, s, launch_moment_split(X, ld, channels, c_pad, t0, n, b.mu_hi, b.mu_lo,
                                                 b.scale_e, b.hi, b.lo, s));
    LAUNCH(K_MOMENT_PRODUCT, s, launch_moment_product(b.hi, b.lo, c_pad, n, b.scale_e, b.partial,
                                                      &b.st->status, s));
    LAUNCH(K_MOMENT_SUM, s, launch_moment_sum(b.partial, c_pad, channels, n, cen, b.sum, b.mu_hi,
                                              b.mu_lo, accumulate ? 1 : 0, out, s));
    MomentStatus h{};
    CUDA_OK(cudaMemcpyAsync(&h, b.st, sizeof(MomentStatus), cudaMemcpyDeviceToHost, s));
    CUDA_OK(cudaStreamSynchronize(s));
    if (h.status & kStatusNonFinite) return HDBMST_ERR_NONFINITE;
    if (h.status & kStatusTimeout) return HDBMST_ERR_TIMEOUT;
    return HDBMST_OK;
}

int hdbmst_last_assign_moved(int64_t *moved, int max_rounds) {
    const int r = static_cast<int>(g_assign_moved.size());
    for (int i = 0; i < std::min(r, max_rounds); ++i)
        if (moved) moved[i] = g_assign_moved[i];
    return r;
}

int hdbmst_set_engine(int engine) {
    const int prev = g_engine;
    if (engine == HDBMST_ENGINE_AUTO || engine == HDBMST_ENGINE_SIMT ||
        engine == HDBMST_ENGINE_TENSOR || engine == HDBMST_ENGINE_TF32)
        g_engine = engine;
    return prev;
}

int64_t hdbmst_set_scan_list_cap(int64_t cap) {
    const int64_t prev = g_list_cap;
    g_list_cap = cap > 0 ? cap : 0;
    return prev;
}

hdbmst_status hdbmst_test_set_tc_hooks(uint64_t wait_ns, int withhold_first_slab) {
    const unsigned long long ns = wait_ns ? wait_ns : tc::kWaitNs;
    const int w = withhold_first_slab ? 1 : 0;
    cudaError_t e = tc_knn_test_hooks(ns, w);
    if (e == cudaSuccess) e = tc_scan_test_hooks(ns, w);
    if (e == cudaSuccess) e = tc_sym_test_hooks(ns, w);
    if (e == cudaSuccess) e = moment_test_hooks(ns, w);
    return e == cudaSuccess ? HDBMST_OK : cuda_fail(e);
}

hdbmst_status hdbmst_test_tmem_max(float *out) {
    if (!out) return HDBMST_ERR_ARG;
    if (cudaSuccess != tc_tmem_max_probe(out, nullptr)) return HDBMST_ERR_CUDA;
    return cudaSuccess == cudaStreamSynchronize(nullptr) ? HDBMST_OK : HDBMST_ERR_CUDA;
}

void hdbmst_test_set_mst_caps(int max_rounds, int max_jump_launches) {
    g_test_max_rounds = std::max(0, max_rounds);
    g_test_jump_launches = std::max(0, max_jump_launches);
}

int hdbmst_set_scan_pruning(int on) {
    const int prev = g_sym_prune ? 1 : 0;
    g_sym_prune = on != 0;
    return prev;
}

int hdbmst_set_scan_form(int form) {
    const int prev = g_scan_form;
    if (form == HDBMST_SCAN_AUTO || form == HDBMST_SCAN_ONE_SIDED || form == HDBMST_SCAN_SYMMETRIC)
        g_scan_form = form;
    return prev;
}

uint64_t hdbmst_launch_count(void) { return g_launches.load(); }

void hdbmst_profile_enable(int on) {
    g_prof = on != 0;
    // create the events up front: creating them between launches would stall
    // the host, and with it the device, inside the timed work
    if (g_prof)
        while (g_pool.size() + g_recs.size() * 2 < 8192) {
            cudaEvent_t e = nullptr;
            if (cudaEventCreate(&e) != cudaSuccess) break;
            g_pool.push_back(e);
        }
}

int hdbmst_profile_read(double *total_ms, int64_t *launches, int max_kernels) {
    double ms[K_COUNT] = {0};
    int64_t cnt[K_COUNT] = {0};
    for (ProfRec &r : g_recs) {
        if (r.b) {
            float t = 0.f;
            if (cudaEventSynchronize(r.b) == cudaSuccess &&
                cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess) {
                ms[r.id] += t;
                cnt[r.id] += 1;
            }
            g_pool.push_back(r.b);
        }
        g_pool.push_back(r.a);
    }
    g_recs.clear();
    for (int i = 0; i < std::min(max_kernels, static_cast<int>(K_COUNT)); ++i) {
        if (total_ms) total_ms[i] = ms[i];
        if (launches) launches[i] = cnt[i];
    }
    return K_COUNT;
}

int hdbmst_last_mst_rounds(int64_t *active, int64_t *edges, int64_t *exact_rows,
                           int max_rounds) {
    const int r = static_cast<int>(g_round_active.size());
    for (int i = 0; i < std::min(r, max_rounds); ++i) {
        if (active) active[i] = g_round_active[i];
        if (edges) edges[i] = g_round_edges[i];
        if (exact_rows) exact_rows[i] = g_round_exact[i];
    }
    return r;
}

int hdbmst_last_mst_symmetric(int64_t *recorded, int max_rounds) {
    const int r = static_cast<int>(g_round_sym.size());
    for (int i = 0; i < std::min(r, max_rounds); ++i)
        if (recorded) recorded[i] = g_round_sym[i];
    return r;
}

int64_t hdbmst_last_knn_exact_rows(void) { return g_knn_exact_rows; }

int64_t hdbmst_last_knn_tile_pairs(void) { return g_knn_tile_pairs; }

int64_t hdbmst_last_mst_scan_pairs(void) { return g_mst_scan_pairs; }

const char *hdbmst_profile_kernel_name(int i) {
    return (i >= 0 && i < K_COUNT) ? kKernelNames[i] : "";
}

}  // extern "C"
