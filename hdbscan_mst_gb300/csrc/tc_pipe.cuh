// The warp-specialized tensor-core distance-tile pipeline shared by the k-NN
// search and the Boruvka scan.
//
// One CTA per SM owns 128 rows (the A operand, resident) and a sequence of
// 128-column tiles (the B operand, streamed).  Dot products use three TF32
// passes (hi.hi + hi.lo + lo.hi, see tc.cuh); the operands come from
// point-major [rows][dk] float32 arrays of hi (raw) and lo parts through 2-D
// TMA tensor maps with 128-byte swizzle, dk = 32 or 64.
//
// Roles: warps 0 .. E-1 are the caller's epilogue, warp E the TMA producer
// (one lane), warp E+1 the MMA issuer (one lane, also owns the TMEM
// allocation).  Stages: a 4-deep ring of 32-feature slabs (full/empty
// mbarriers) and four 128-column TMEM accumulators (afull/aempty), all 512
// columns of TMEM.  The epilogue warps form E / 4 groups of four (one warp per
// 32-lane TMEM quadrant); group g takes the tiles t with t % (E / 4) = g,
// whole, so each warp has E / 4 tile periods for one tile and the latency of
// its chain (TMEM load, norms, selection) hides behind the other groups' work.
// Every wait is bounded; the first that gives up sets S.abort, every role
// winds down, and tc_teardown drains and frees TMEM.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace hdbmst {
namespace tc {

constexpr int kStages = 4;
constexpr int kAcc = 4;  // TMEM accumulators of kCols columns
constexpr uint32_t kSlabTile = kRows * kSlabBytes;  // 16 KB: one slab of 128 rows
// dynamic shared memory: resident rows (hi + lo, up to 2 slabs) + the ring
constexpr size_t kPipeSmem = (2 * 2 + 2 * kStages) * kSlabTile + 1024;

struct PipeMaps {
    CUtensorMap a_hi, a_lo, b_hi, b_lo;
};

struct PipeSmem {
    uint64_t full[kStages], empty[kStages], afull[kAcc], aempty[kAcc], abar;
    uint32_t tmem_base;
    int abort;
};

// The column tiles of a CTA: [ct_begin, ct_end) without [skip_lo, skip_hi).
struct TileSeq {
    int ct_begin, n, s_lo, gap;
    __device__ TileSeq(int begin, int end, int skip_lo, int skip_hi) {
        ct_begin = begin;
        s_lo = min(max(skip_lo, begin), end);
        const int s_hi = max(min(skip_hi, end), s_lo);
        gap = s_hi - s_lo;
        n = max(end - begin - gap, 0);
    }
    __device__ int at(int k) const {
        const int t = ct_begin + k;
        return t >= s_lo ? t + gap : t;
    }
};

__device__ __forceinline__ uint8_t *pipe_base(uint8_t *smem_raw) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
}

// Barrier initialisation and TMEM allocation; all threads, before anything else.
template <int kEpiWarps>
__device__ __forceinline__ void tc_setup(PipeSmem &S) {
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], 1);
        }
        for (int i = 0; i < kAcc; ++i) {
            mbar_init(&S.afull[i], 1);
            mbar_init(&S.aempty[i], 4 * 32);  // the four warps of one group
        }
        mbar_init(&S.abar, 1);
        S.abort = 0;
        fence_mbar_init();
    }
    static_assert(kAcc % (kEpiWarps / 4) == 0, "each accumulator belongs to one group");
    if (warp == kEpiWarps + 1) tmem_alloc(&S.tmem_base, kAcc * kCols);
}

// Producer and MMA roles (warps E and E+1); epilogue warps return at once.
// a_row: first row of the A operand in its tensor map.
template <int kEpiWarps>
__device__ __forceinline__ void tc_produce_and_multiply(const PipeMaps &M, PipeSmem &S,
                                                        uint32_t sbase, int dk, int a_row,
                                                        const TileSeq &seq) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slabs = dk / kSlab;
    const uint32_t a_hi = sbase, a_lo = sbase + slabs * kSlabTile;
    const uint32_t ring = sbase + 2 * slabs * kSlabTile;
    if (warp == kEpiWarps && lane == 0) {
        mbar_expect_tx(&S.abar, 2 * slabs * kSlabTile);
        for (int s = 0; s < slabs; ++s) {
            tma_load_2d(a_hi + s * kSlabTile, &M.a_hi, s * kSlab, a_row, &S.abar);
            tma_load_2d(a_lo + s * kSlabTile, &M.a_lo, s * kSlab, a_row, &S.abar);
        }
        int it = 0;
        for (int t = 0; t < seq.n; ++t) {
            const int col0 = seq.at(t) * kCols;
            for (int s = 0; s < slabs; ++s, ++it) {
                const int st = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                if (!mbar_wait<kSleepProducer>(&S.empty[st], ph ^ 1) ||
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
    } else if (warp == kEpiWarps + 1 && lane == 0) {
        const uint32_t idesc = instr_desc(kRows, kCols);
        const uint32_t tmem = S.tmem_base;
        bool ok = mbar_wait<kSleepMma>(&S.abar, 0);
        int it = 0;
        for (int t = 0; t < seq.n && ok; ++t) {
            const int acc = t % kAcc;
            ok = mbar_wait<kSleepMma>(&S.aempty[acc], ((t / kAcc) & 1) ^ 1) &&
                 !*(volatile int *)&S.abort;
            if (!ok) break;
            fence_after();
            const uint32_t d = tmem + static_cast<uint32_t>(acc * kCols);
            for (int s = 0; s < slabs; ++s, ++it) {
                const int st = it % kStages;
                ok = mbar_wait<kSleepMma>(&S.full[st], (it / kStages) & 1);
                if (!ok) break;
                fence_after();
                const uint32_t hi = ring + st * 2 * kSlabTile;
#pragma unroll
                for (int kk = 0; kk < kSlab / 8; ++kk) {
                    const uint32_t off = kk * 32;
                    const uint64_t ah = smem_desc(a_hi + s * kSlabTile + off);
                    const uint64_t al = smem_desc(a_lo + s * kSlabTile + off);
                    const uint64_t bh = smem_desc(hi + off), bl = smem_desc(hi + kSlabTile + off);
                    mma_tf32(d, ah, bh, idesc, (s > 0 || kk > 0) ? 1u : 0u);
                    mma_tf32(d, ah, bl, idesc, 1u);
                    mma_tf32(d, al, bh, idesc, 1u);
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
// every tile of its group, waits for the tile's accumulator and calls
// consume(tmem_addr, col0) with the TMEM address of this thread's lane at the
// tile's first column and the tile's first global column; then hands the
// accumulator back.
template <int kEpiWarps, class Consume>
__device__ __forceinline__ void tc_epilogue_loop(PipeSmem &S, const TileSeq &seq,
                                                 Consume &&consume) {
    constexpr int kGroups = kEpiWarps / 4;
    const int warp = threadIdx.x >> 5;
    const int group = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tmem = S.tmem_base;
    for (int t = group; t < seq.n; t += kGroups) {
        const int acc = t % kAcc;
        const bool w = mbar_wait<kSleepEpilogue>(&S.afull[acc], (t / kAcc) & 1);
        if (!w) S.abort = 1;
        // a warp leaves together: tcgen05.ld is warp-collective
        if (__any_sync(0xffffffffu, !w || *(volatile int *)&S.abort)) break;
        fence_after();
        consume(tmem + static_cast<uint32_t>(acc * kCols) + lane_base, seq.at(t) * kCols);
        fence_before();
        mbar_arrive(&S.aempty[acc]);
    }
}

// All threads, last: report a give-up, drain what may still be in flight
// (bounded), free TMEM.
template <int kEpiWarps>
__device__ __forceinline__ void tc_teardown(PipeSmem &S, unsigned *status) {
    const int tid = threadIdx.x, warp = tid >> 5;
    fence_before();
    __syncthreads();
    if (S.abort) {
        if (tid == 0) {
            atomicOr(status, kStatusTimeout);
            for (int i = 0; i < kAcc; ++i) mbar_wait<kSleepProducer>(&S.afull[i], 0);
            for (int i = 0; i < kStages; ++i) mbar_wait<kSleepProducer>(&S.full[i], 0);
        }
        __syncthreads();
    }
    fence_after();
    if (warp == kEpiWarps + 1) tmem_free(S.tmem_base, kAcc * kCols);
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
