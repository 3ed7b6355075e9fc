// The warp-specialized tensor-core distance-tile pipeline shared by the k-NN
// search and the Boruvka scan.
//
// One CTA per SM owns 128 rows (the A operand, resident in TMEM) and a
// sequence of 64-column tiles (the B operand, streamed through shared
// memory in 128-column slabs, each shared by the two tiles it holds).  Dot products use three TF32 passes (hi.hi + hi.lo + lo.hi, see
// tc.cuh); the operands come from point-major [rows][dk] float32 arrays of hi
// (raw) and lo parts, dk = 32 or 64: the first epilogue group writes the A
// rows into TMEM columns [0, 2 dk) once, and B arrives through 2-D TMA tensor
// maps with 128-byte swizzle.  With A in TMEM the tensor core reads only B
// from shared memory, half the bytes per MMA.
//
// Roles: warps 0 .. E-1 are the caller's epilogue, warp E the TMA producer
// (one lane), warps E+1 .. E+G the MMA issuers, G = E / 4 (one lane each; E+1
// also owns the TMEM allocation).  Tile t belongs to group and issuer t % G: a
// single issuing thread is a serial chain of barrier tests, fences, descriptor
// arithmetic and MMA issues that falls behind the tensor core (measured: 82
// cycles of thread time per 64-cycle MMA), several keep its queue fed.  Each
// group has two accumulators that its tiles alternate between, so the MMAs
// of a group's next tile run while the group selects from the current one;
// each issuer owns its group's accumulators and its share of the ring, so
// every barrier is used in order by one thread and its phase parity cannot
// alias.  Stages: a 6-deep ring of 32-feature slabs (full/empty
// mbarriers) and two 64-column TMEM accumulators per epilogue group
// (afull/aempty) after the A columns, in a 512-column allocation.  The epilogue warps
// form E / 4 groups of four (one warp per 32-lane TMEM quadrant); group g
// takes the tiles t with t % (E / 4) = g, whole, so each warp has E / 4 tile
// periods for one tile and the latency of its chain (TMEM load, column data,
// selection) hides behind the other groups' work.  Each epilogue warp
// prefetches the column data of its next tile with cp.async while the tile
// before it is multiplied.
// Wide rows (kWide, 64 < dk <= 192): the A hi parts alone fill TMEM columns
// [0, dk), the A lo parts sit in shared memory (TMA, once per CTA) ahead of a
// 3-stage ring, the lo.hi MMAs read both operands from shared memory, and two
// epilogue groups keep their accumulators in TMEM columns [256, 512).
//
// Every wait is bounded; the first that gives up sets S.abort, every role
// winds down, and tc_teardown drains and frees TMEM.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace hdbmst {
namespace tc {

constexpr int kStages = 6;       // ring slabs (kWide: kWideStages)
constexpr int kWideStages = 3;
constexpr int kSmallStages = 2;
constexpr int kWideDkMax = 192;
constexpr int kTileCols = 64;   // columns of a tile (MMA N); a ring slab holds kCols = 2 tiles
constexpr int kAccPerGroup = 2;

// Ring slot of slab s of the 128-column block at position h of the sequence:
// stages are used in order (u counts slabs) and each use is consumed by the
// two tiles 2h and 2h + 1.  With G = 2 or 3 issuers and a ring of 6 slabs
// (dk = 64: 3 blocks, dk = 32: 6 blocks) the tiles of block h - ring depth
// belong to the same two issuers as those of block h, so an issuer that waits
// on a stage's use has waited on its previous use itself and the phase parity
// cannot alias.
template <int kSt>
struct Slot {
    int st;
    uint32_t parity;
    __device__ Slot(int h, int s, int slabs) {
        const int u = h * slabs + s;
        st = u % kSt;
        parity = static_cast<uint32_t>(u / kSt) & 1u;
    }
};

// kSmall: a narrow pipeline for two CTAs per SM (a 2-slab ring, 256 TMEM
// columns: A in [0, 128), one group's two accumulators in [128, 256)).
template <bool kWide, bool kSmall = false>
struct PipeShape {
    static constexpr int kSt = kWide ? kWideStages : (kSmall ? kSmallStages : kStages);
    static constexpr uint32_t kAccBase = kWide ? 256u : 128u;  // first accumulator column
    static constexpr uint32_t kCols = kSmall ? 256u : 512u;    // the TMEM allocation
};
constexpr int kAccMax = 6;          // TMEM accumulators of kTileCols columns
constexpr uint32_t kAccBase = 128;  // TMEM columns [0, 2 dk) hold A hi and lo
constexpr uint32_t kTmemCols = 512; // the allocation

// Epilogue groups = MMA issuers; each owns kAccPerGroup accumulators.
template <int kEpiWarps>
__host__ __device__ constexpr int acc_count() {
    return kEpiWarps / 4;
}
constexpr uint32_t kSlabTile = kCols * kSlabBytes;  // 16 KB: one slab of 128 columns
// dynamic shared memory: the ring (a stage holds one slab, hi and lo); kWide:
// the A lo slabs, then the ring
constexpr size_t kPipeSmem = 2 * kStages * kSlabTile + 1024;
constexpr size_t kWidePipeSmem = (kWideDkMax / kSlab + 2 * kWideStages) * kSlabTile + 1024;
constexpr size_t kSmallPipeSmem = 2 * kSmallStages * kSlabTile + 1024;

// Accumulator of tile t: group j = t % G alternates between its two.
template <int G>
struct AccSlot {
    int acc;
    uint32_t parity;  // phase parity of the tile's use of the accumulator
    __device__ AccSlot(int t) {
        const int lt = t / G;
        acc = (t % G) * kAccPerGroup + lt % kAccPerGroup;
        parity = static_cast<uint32_t>(lt / kAccPerGroup) & 1u;
    }
};

struct PipeMaps {
    CUtensorMap b_hi, b_lo;
    CUtensorMap a_lo;  // kWide only: the A rows' lo parts
};

struct PipeSmem {
    uint64_t full[kStages], empty[kStages], afull[kAccMax], aempty[kAccMax], abar;
    uint32_t tmem_base;
    int abort;
};

// The column tiles of a CTA: [ct_begin, ct_end) without [skip_lo, skip_hi),
// optionally rotated: position t maps to (t + rot) mod wrap (wrap > 0), so a
// sweep can start anywhere and wrap around (rot and wrap even: whole blocks).
// With a block list, position t is tile t % 2 of the 128-column block
// list[t / 2] (n = twice the list's length).
struct TileSeq {
    int ct_begin, n, s_lo, gap, rot = 0, wrap = 0;
    const int *list = nullptr;
    __device__ TileSeq(int begin, int end, int skip_lo, int skip_hi) {
        ct_begin = begin;
        s_lo = min(max(skip_lo, begin), end);
        const int s_hi = max(min(skip_hi, end), s_lo);
        gap = s_hi - s_lo;
        n = max(end - begin - gap, 0);
    }
    __device__ int at(int k) const {
        if (list) return list[k >> 1] * 2 + (k & 1);  // shared or global memory
        int t = ct_begin + k;
        t = t >= s_lo ? t + gap : t;
        if (wrap > 0) {
            t += rot;
            if (t >= wrap) t -= wrap;
        }
        return t;
    }
};

__device__ __forceinline__ uint8_t *pipe_base(uint8_t *smem_raw) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
}

// Barrier initialisation and TMEM allocation; all threads, before anything else.
template <int kEpiWarps, bool kWide = false, bool kSmall = false>
__device__ __forceinline__ void tc_setup(PipeSmem &S) {
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], 2);  // both tiles of the block
        }
        for (int i = 0; i < acc_count<kEpiWarps>() * kAccPerGroup; ++i) {
            mbar_init(&S.afull[i], 1);
            mbar_init(&S.aempty[i], 4 * 32);  // the four warps of one group
        }
        // warps 0 .. 3 once A is in TMEM (+ the producer's TMA of A lo)
        mbar_init(&S.abar, 4 * 32 + (kWide ? 1 : 0));
        S.abort = 0;
        fence_mbar_init();
    }
    static_assert(acc_count<kEpiWarps>() * kAccPerGroup <= kAccMax, "accumulators");
    static_assert(kAccBase + kAccMax * kTileCols <= kTmemCols, "TMEM budget");
    static_assert(!kSmall || (!kWide && kAccBase + acc_count<kEpiWarps>() * kAccPerGroup * kTileCols <=
                                            PipeShape<false, true>::kCols),
                  "TMEM budget, small pipeline");
    static_assert(!kWide || (acc_count<kEpiWarps>() * kAccPerGroup * kTileCols + 256 <= kTmemCols &&
                             kWideDkMax <= 256), "TMEM budget, wide rows");
    if (warp == kEpiWarps + 1) tmem_alloc(&S.tmem_base, PipeShape<kWide, kSmall>::kCols);
}

// The A operand into TMEM, by the first epilogue group (warps 0 .. 3, one per
// 32-lane quadrant): thread (w, lane) copies row 32 w + lane of the CTA's row
// block - hi parts to columns [0, dk), lo parts to [dk, 2 dk) - then arrives
// on S.abar.  rows: point-major [..][dk] arrays, row0: the block's first row.
// kBoth: A's lo parts go to TMEM too (after the hi parts), as everywhere but
// the wide TF32 rows, whose lo parts the producer loads into shared memory.
template <bool kWide = false, bool kBoth = !kWide>
__device__ __forceinline__ void tc_load_a(PipeSmem &S, const float *a_hi, const float *a_lo,
                                          int64_t row0, int dk) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t taddr = S.tmem_base + (static_cast<uint32_t>(warp * 32) << 16);
    const int64_t off = (row0 + warp * 32 + lane) * dk;
#pragma unroll 1
    for (int h = 0; h < (kBoth ? 2 : 1); ++h) {
        const float *src = (h ? a_lo : a_hi) + off;
#pragma unroll 1
        for (int c = 0; c < dk; c += 32) {
            float v[32];
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
                const float4 x = __ldg(reinterpret_cast<const float4 *>(src + c + j4 * 4));
                v[j4 * 4 + 0] = x.x;
                v[j4 * 4 + 1] = x.y;
                v[j4 * 4 + 2] = x.z;
                v[j4 * 4 + 3] = x.w;
            }
            tmem_st32(taddr + static_cast<uint32_t>(h * dk + c), v);
        }
    }
    tmem_wait_st();
    fence_before();
    mbar_arrive(&S.abar);
}

// Producer and MMA roles (warps E, E+1, E+2); epilogue warps return at once.
// kF16: the operands are the two-part FP16 halves (tc.cuh), two per 32-bit
// word; dk then counts words, and the K steps, slabs, TMEM columns and
// descriptors are those of the TF32 form on dk words, only the MMA kind
// differs (K = 16 halves per MMA instead of 8 floats: the same 32 bytes).
template <int kEpiWarps, bool kWide = false, bool kF16 = false, bool kSmall = false>
__device__ __forceinline__ void tc_produce_and_multiply(const PipeMaps &M, PipeSmem &S,
                                                        uint32_t sbase, int dk, int a_row,
                                                        const TileSeq &seq) {
    using Sh = PipeShape<kWide, kSmall>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slabs = dk / kSlab;
    const uint32_t alo = sbase;  // kWide: A lo slabs
    const uint32_t ring = sbase + (kWide ? static_cast<uint32_t>(slabs) * kSlabTile : 0u);
    constexpr int kAcc = acc_count<kEpiWarps>();  // = issuers = epilogue groups
    // one issuer (kSmall) owns every stage, so no phase parity can alias
    static_assert(kWide ? kAcc == 2
                        : kSmall ? kAcc == 1 : ((kAcc == 2 || kAcc == 3) && kStages == 6),
                  "see Slot");
    if (warp == kEpiWarps && lane == 0) {
        if constexpr (kWide && !kF16) {
            mbar_expect_tx(&S.abar, static_cast<uint32_t>(slabs) * kSlabTile);
            for (int s = 0; s < slabs; ++s)
                tma_load_2d(alo + s * kSlabTile, &M.a_lo, s * kSlab, a_row, &S.abar);
        } else if constexpr (kWide) {
            // wide FP16 rows: both A parts are in TMEM (tc_load_a); the
            // producer's arrival that A's lo parts would have completed
            mbar_arrive(&S.abar);
        }
        const bool withhold = *reinterpret_cast<volatile int *>(&g_withhold_first_slab) != 0;
        for (int h = 0; 2 * h < seq.n; ++h) {
            const int col0 = seq.at(2 * h) * kTileCols;
            for (int s = 0; s < slabs; ++s) {
                if (withhold && h == 0 && s == 0) continue;  // test hook: never arrives
                const Slot<Sh::kSt> slot(h, s, slabs);
                const int st = slot.st;
                if (!mbar_wait<kSleepProducer>(&S.empty[st], slot.parity ^ 1) ||
                    *(volatile int *)&S.abort) {
                    S.abort = 1;
                    return;
                }
                const uint32_t hi = ring + st * 2 * kSlabTile;
                mbar_expect_tx(&S.full[st], 2 * kSlabTile);
                tma_load_2d(hi, &M.b_hi, s * kSlab, col0, &S.full[st]);
                tma_load_2d(hi + kSlabTile, &M.b_lo, s * kSlab, col0, &S.full[st]);
            }
        }
    } else if (warp > kEpiWarps && warp <= kEpiWarps + kAcc && lane == 0) {
        const int issuer = warp - kEpiWarps - 1;
        const uint32_t idesc =
            kF16 ? instr_desc_f16(kRows, kTileCols) : instr_desc(kRows, kTileCols);
        const uint32_t tmem = S.tmem_base;
        bool ok = mbar_wait<kSleepMma>(&S.abar, 0);
        if (ok) fence_after();
        for (int t = issuer; t < seq.n && ok; t += kAcc) {
            const AccSlot<kAcc> as(t);
            const int acc = as.acc;
            ok = mbar_wait<kSleepMma>(&S.aempty[acc], as.parity ^ 1) &&
                 !*(volatile int *)&S.abort;
            if (!ok) break;
            fence_after();
            const uint32_t d = tmem + Sh::kAccBase + static_cast<uint32_t>(acc * kTileCols);
            for (int s = 0; s < slabs; ++s) {
                const Slot<Sh::kSt> slot(t >> 1, s, slabs);
                const int st = slot.st;
                ok = mbar_wait<kSleepMma>(&S.full[st], slot.parity);
                if (!ok) break;
                fence_after();
                // The issuing thread is a serial chain, so keep it short: the
                // descriptors of the slab's K steps are the slab's first one
                // plus 32 bytes (2 in the address field) per step; the odd tile
                // of a block starts 64 rows (8 KB) into the slab.
                const uint64_t bh = smem_desc(ring + st * 2 * kSlabTile + (t & 1) * (kSlabTile / 2));
                const uint64_t bl = bh + (kSlabTile >> 4);
                const uint32_t ah = tmem + static_cast<uint32_t>(s * kSlab), al = ah + dk;
                if constexpr (kWide && !kF16) {
                    // A lo from shared memory: its slab's descriptor, + 2 per K step
                    const uint64_t als = smem_desc(alo + s * kSlabTile);
                    mma_tf32_ts(d, ah, bh, idesc, s > 0 ? 1u : 0u);
                    mma_tf32_ts(d, ah, bl, idesc, 1u);
                    mma_tf32(d, als, bh, idesc, 1u);
#pragma unroll
                    for (int kk = 1; kk < kSlab / 8; ++kk) {
                        mma_tf32_ts(d, ah + kk * 8, bh + 2 * kk, idesc, 1u);
                        mma_tf32_ts(d, ah + kk * 8, bl + 2 * kk, idesc, 1u);
                        mma_tf32(d, als + 2 * kk, bh + 2 * kk, idesc, 1u);
                    }
                } else if constexpr (kF16) {
                    // A hi in TMEM columns [0, dk), A lo in [dk, 2 dk)
                    mma_f16_ts(d, ah, bh, idesc, s > 0 ? 1u : 0u);
                    mma_f16_ts(d, ah, bl, idesc, 1u);
                    mma_f16_ts(d, al, bh, idesc, 1u);
#pragma unroll
                    for (int kk = 1; kk < kSlab / 8; ++kk) {
                        mma_f16_ts(d, ah + kk * 8, bh + 2 * kk, idesc, 1u);
                        mma_f16_ts(d, ah + kk * 8, bl + 2 * kk, idesc, 1u);
                        mma_f16_ts(d, al + kk * 8, bh + 2 * kk, idesc, 1u);
                    }
                } else {
                    mma_tf32_ts(d, ah, bh, idesc, s > 0 ? 1u : 0u);
                    mma_tf32_ts(d, ah, bl, idesc, 1u);
                    mma_tf32_ts(d, al, bh, idesc, 1u);
#pragma unroll
                    for (int kk = 1; kk < kSlab / 8; ++kk) {
                        mma_tf32_ts(d, ah + kk * 8, bh + 2 * kk, idesc, 1u);
                        mma_tf32_ts(d, ah + kk * 8, bl + 2 * kk, idesc, 1u);
                        mma_tf32_ts(d, al + kk * 8, bh + 2 * kk, idesc, 1u);
                    }
                }
                mma_commit(&S.empty[st]);
            }
            if (!ok) break;
            mma_commit(&S.afull[acc]);
        }
        if (!ok) S.abort = 1;
    }
}

// Epilogue loop of warp w < E (group w / 4, TMEM lanes 32 (w % 4) ..): for
// every tile of its group, calls prefetch(col0, buf) for the group's next tile
// (the warp issues cp.async copies of that tile's column data into its buffer
// buf of two), waits for the tile's accumulator and its own copies, and calls
// consume(tmem_addr, col0, buf) with the TMEM address of this thread's lane at
// the tile's first column, the tile's first global column and the buffer
// holding its column data; then hands the accumulator back.
template <int kEpiWarps, bool kWide = false, bool kSmall = false, class Prefetch, class Consume>
__device__ __forceinline__ void tc_epilogue_loop(PipeSmem &S, const TileSeq &seq,
                                                 Prefetch &&prefetch, Consume &&consume) {
    using Sh = PipeShape<kWide, kSmall>;
    constexpr int kGroups = kEpiWarps / 4;
    constexpr int kAcc = acc_count<kEpiWarps>();
    const int warp = threadIdx.x >> 5;
    const int group = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tmem = S.tmem_base;
    if (group < seq.n) prefetch(seq.at(group) * kTileCols, 0);
    cp_async_commit();
    for (int t = group, k = 0; t < seq.n; t += kGroups, ++k) {
        if (t + kGroups < seq.n) prefetch(seq.at(t + kGroups) * kTileCols, (k + 1) & 1);
        cp_async_commit();
        const AccSlot<kAcc> as(t);
        const int acc = as.acc;
        const bool w = mbar_wait<kSleepEpilogue>(&S.afull[acc], as.parity);
        if (!w) S.abort = 1;
        // a warp leaves together: tcgen05.ld is warp-collective
        if (__any_sync(0xffffffffu, !w || *(volatile int *)&S.abort)) break;
        cp_async_wait_one();  // this tile's column data (all but the newest group)
        __syncwarp();
        fence_after();
        consume(tmem + Sh::kAccBase + static_cast<uint32_t>(acc * kTileCols) + lane_base,
                seq.at(t) * kTileCols, k & 1);
        fence_before();
        __syncwarp();  // the buffer is refilled two tiles later
        mbar_arrive(&S.aempty[acc]);
    }
    cp_async_wait_all();
}

// All threads, last: report a give-up, drain what may still be in flight
// (bounded), free TMEM.
template <int kEpiWarps, bool kWide = false, bool kSmall = false>
__device__ __forceinline__ void tc_teardown(PipeSmem &S, unsigned *status) {
    const int tid = threadIdx.x, warp = tid >> 5;
    fence_before();
    __syncthreads();
    if (S.abort) {
        if (tid == 0) {
            atomicOr(status, kStatusTimeout);
            for (int i = 0; i < acc_count<kEpiWarps>() * kAccPerGroup; ++i)
                mbar_wait<kSleepProducer>(&S.afull[i], 0);
            for (int i = 0; i < PipeShape<kWide, kSmall>::kSt; ++i)
                mbar_wait<kSleepProducer>(&S.full[i], 0);
        }
        __syncthreads();
    }
    fence_after();
    if (warp == kEpiWarps + 1) tmem_free(S.tmem_base, PipeShape<kWide, kSmall>::kCols);
}

// Named barrier over the epilogue warps only (barrier 1).
template <int kEpiWarps>
__device__ __forceinline__ void epilogue_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
}

// Host: a 2-D map of a point-major [rows][dk] float32 array in boxes of 128
// rows x 32 features with 128-byte swizzle (tc_pipe.cu).
bool make_point_map(CUtensorMap *m, const float *ptr, int64_t rows, int dk);
bool tensor_maps_available();

}  // namespace tc
}  // namespace hdbmst
