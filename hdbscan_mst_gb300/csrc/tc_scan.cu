// K6 on the tensor cores: the Boruvka scan with tcgen05 TF32 MMAs.
//
// Same contract as mst_scan_kernel (page "HDBSCAN", gpu/hdbscan, "Exact
// shortcuts": only the points the shortcuts leave are scanned against all
// others, over a list of active points).  Rows are the active points and
// columns all points, both grouped by component; a row tile whose rows share
// one component skips the column tiles inside that component.  Per (row,
// column) the epilogue forms t = |b|^2 - 2 a.b and ranks the pair by
//     v = max(t, core_b^2 - |a|^2, core_a^2 - |a|^2)  ~  w(a, b)^2 - |a|^2
// over columns of other components.  The epilogue warps form E / 4 groups
// that take every (E / 4)-th tile whole, so each row has one list per group:
// its 4 best (v, point) keys in registers and the least v it dropped; the
// groups of a row filter against the least of their published 4th values.
// Columns of the row's own component (one run of the grouped order) are
// masked out by position.  At the end the lists merge into the row's 4 best
// and a threshold tau that every other column reaches or exceeds, which
// mst_refine_kernel re-evaluates exactly and proves (this engine's rounding
// bound) - the same output as the FFMA scan.
#include <climits>
#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tc_pipe.cuh"

namespace hdbmst {

namespace {

using namespace tc;

constexpr int kKeep = 4;
constexpr int kEpiWarps = 12;
constexpr int kParts = kEpiWarps / 4;
constexpr int kScanThreads = (kEpiWarps + 1 + kEpiWarps / 4) * 32;  // + producer + MMA warps

struct TcScanParams {
    PipeMaps maps;             // B: grouped columns, point-major [rows][dk]
    const float *a_hi, *a_lo;  // A: active rows, point-major [rows][dk]
    ScanArgs a;
};

__shared__ float s_row_thr[kParts][kRows];  // per group and row: its 4th kept v
__shared__ int s_rcomp[kRows];
// per warp, two tiles: the columns' norms
__shared__ float4 s_cnorm[kEpiWarps][2][kTileCols / 4];
__shared__ float2 s_cnmin[kEpiWarps][2];  // per warp, two tiles: each batch's least norm

__device__ __forceinline__ void keep_insert(unsigned long long (&k)[kKeep], unsigned long long key,
                                            float &dropped) {
    if (key < k[kKeep - 1]) {
        if (k[kKeep - 1] != kNoKey)
            dropped = fminf(dropped, order_float(static_cast<unsigned>(k[kKeep - 1] >> 32)));
        k[kKeep - 1] = key;
#pragma unroll
        for (int p = kKeep - 1; p > 0; --p) {
            const unsigned long long lo = min(k[p - 1], k[p]), hi = max(k[p - 1], k[p]);
            k[p - 1] = lo;
            k[p] = hi;
        }
    } else {
        dropped = fminf(dropped, order_float(static_cast<unsigned>(key >> 32)));
    }
}

__device__ __forceinline__ float key_v(unsigned long long k) {
    return k == kNoKey ? INFINITY : order_float(static_cast<unsigned>(k >> 32));
}

template <bool kF16>
__global__ void __launch_bounds__(kScanThreads, 1) tc_scan_kernel(const __grid_constant__ TcScanParams P) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ PipeSmem S;
    const ScanArgs &a = P.a;
    uint8_t *base = pipe_base(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = blockIdx.x * kRows;
    const int split = blockIdx.y;
    constexpr int kSub = kCols / kTileCols;  // pipeline tiles per 128-column tile
    const int ct_begin = split * a.tiles_per_split * kSub;
    const int ct_end = min(split * a.tiles_per_split + a.tiles_per_split, a.col_tiles) * kSub;

    for (int i = tid; i < kParts * kRows; i += blockDim.x) (&s_row_thr[0][0])[i] = INFINITY;
    if (tid < kRows) s_rcomp[tid] = r0 + tid < a.na ? a.act_comp[r0 + tid] : -1;
    tc_setup<kEpiWarps>(S);
    fence_before();
    __syncthreads();
    fence_after();
    // rows all in one component: skip the column tiles wholly inside it
    const bool uniform =
        __syncthreads_and(tid >= kRows || r0 + tid >= a.na || s_rcomp[tid] == s_rcomp[0]);
    int skip_lo = 0, skip_hi = 0;
    if (uniform) {
        const int C = s_rcomp[0];
        const int c0 = a.comp_start[C], c1 = c0 + a.comp_size[C];
        // whole 128-column blocks only: a ring slab serves both its tiles
        skip_lo = (c0 + kCols - 1) / kCols * kSub;
        skip_hi = c1 / kCols * kSub;
    }
    const TileSeq seq(ct_begin, ct_end, skip_lo, skip_hi);
    if (tid == 0 && a.tile_pairs)
        atomicAdd(a.tile_pairs, static_cast<unsigned long long>(seq.n) * kTileCols * kRows);
    // the MMA operands: dk floats (TF32), or dk / 2 words of two halves (FP16)
    const int dk_mma = kF16 ? a.dk / 2 : a.dk;
    tc_produce_and_multiply<kEpiWarps, false, kF16>(P.maps, S, smem_u32(base), dk_mma, r0, seq);
    if (warp < 4) tc_load_a(S, P.a_hi, P.a_lo, r0, dk_mma);

    if (warp < kEpiWarps) {
        const int row = (warp & 3) * 32 + lane;
        const int group = warp >> 2;
        const int r = r0 + row;
        const bool valid = r < a.na;
        const float na = valid ? a.act_norm[r] : 0.f;
        const float ca = valid ? a.act_core[r] : 0.f;
        const float ra = __fsub_rn(__fmul_rn(ca, ca), na);
        const int rc = s_rcomp[row];
        unsigned long long keys[kKeep];
#pragma unroll
        for (int p = 0; p < kKeep; ++p) keys[p] = kNoKey;
        float dropped = INFINITY;
        // With the component bound U_C the row needs no column of weight above
        // it: tau0 is the least v a column can have without the refine's proof
        // (with w = U_C) ruling it out, so columns at or above tau0 are dropped
        // and tau0 joins the row's threshold.
        float tau0 = INFINITY;
        if (a.ub && valid) {
            const float uc = __uint_as_float(a.ub[rc]);
            if (uc < INFINITY) {
                // T(U_C) + c (|a|^2 + nb_c) + e0 - |a|^2, rounded up, plus a margin
                // of 2^-20 of its magnitude (the refine's check rounds down)
                const float T = proof_T_up(uc, a.d);
                const float sq = __fadd_ru(__fsqrt_ru(na), __fsqrt_ru(T));
                const float X = __fsub_ru(
                    __fadd_ru(__fadd_ru(T, __fmul_ru(a.err_c, __fadd_ru(na, __fmul_ru(sq, sq)))),
                              *a.e0),
                    na);
                tau0 = __fadd_ru(X, __fmul_ru(__fadd_ru(fabsf(X), __fadd_ru(na, T)), 0x1p-20f));
            }
        }
        // t = |b|^2 - 2 a.b; the FP16 products carry the set's scale 2^2e
        const float kdot = kF16 ? -ldexpf(2.f, -2 * f16_scale_exp(*a.amax_bits)) : -2.f;
        // the row's own component is one run of columns [own_lo, own_hi)
        const int own_lo = valid ? a.comp_start[rc] : 0;
        const int own_hi = valid ? own_lo + a.comp_size[rc] : 0;

        // only the column norms are read per tile; the rare candidate path
        // reads a column's core distance and point index from global memory
        const auto prefetch = [&](int col0, int buf) {
            static_assert(kTileCols == 64, "one 16-byte copy per lane");
            if (lane < 16) cp_async16(&s_cnorm[warp][buf][lane], a.col_norm + col0 + lane * 4);
            else if (lane == 16) cp_async8(&s_cnmin[warp][buf], a.col_nmin + (col0 >> 5));
        };
        tc_epilogue_loop<kEpiWarps>(S, seq, prefetch, [&](uint32_t tbase, int col0, int buf) {
            // the other groups' published 4th values, once per tile (a stale
            // value is only looser)
            float thr_tile = tau0;
#pragma unroll
            for (int q = 0; q < kParts; ++q) thr_tile = fminf(thr_tile, s_row_thr[q][row]);
#pragma unroll 1
            for (int cc = 0; cc < kTileCols / 32; ++cc) {
                const int cb0 = col0 + cc * 32;
                // own-component columns of this batch: bits [blo, bhi)
                const int blo = min(max(own_lo - cb0, 0), 32);
                const int bhi = min(max(own_hi - cb0, 0), 32);
                // skip a batch that is own-component for every row of the
                // warp; the skip must be warp-uniform: tcgen05.ld is collective
                if (__all_sync(0xffffffffu, blo == 0 && bhi == 32)) continue;
                float v[32];
                const float amax = tmem_ld32_max(tbase + cc * 32, v);
                // v >= t, so a batch whose least t does not beat the row's
                // least published 4th value cannot change any list's 4 best;
                // most batches are ruled out by the floor of their t alone
                const float thr = fminf(key_v(keys[kKeep - 1]), thr_tile);
                const float nmin = cc ? s_cnmin[warp][buf].y : s_cnmin[warp][buf].x;
                if (!__any_sync(0xffffffffu, batch_t_floor(kdot, amax, nmin) < thr)) continue;
                expand32(v, &s_cnorm[warp][buf][cc * 8], kdot);
                const float vmin = min32(v);
                if (vmin < thr) {
                    const uint32_t own =
                        bhi > blo ? ((bhi == 32 ? 0u : (1u << bhi)) - (1u << blo)) : 0u;
                    uint32_t mask = below_mask(v, thr) & ~own;
                    if (mask) {
#pragma unroll 1
                        while (mask) {
                            const int j = __ffs(mask) - 1;
                            mask &= mask - 1;
                            const int col = cb0 + j;
                            if (col >= a.n) break;
                            const float cbc = __ldg(a.col_core + col);
                            const float vv = fmaxf(
                                fmaxf(pick32(v, j), __fsub_rn(__fmul_rn(cbc, cbc), na)), ra);
                            const unsigned long long key =
                                (static_cast<unsigned long long>(float_order(vv)) << 32) |
                                static_cast<unsigned>(__ldg(a.col_orig + col));
                            keep_insert(keys, key, dropped);
                        }
                        s_row_thr[group][row] = key_v(keys[kKeep - 1]);
                    }
                }
            }
        });

        // Merge the lists of each row in the idle ring: tau bounds every
        // column not kept - dropped ones directly, filtered ones by the 4th
        // kept value of the group that filtered them.
        unsigned long long *pk =
            reinterpret_cast<unsigned long long *>(base);
        float *pt = reinterpret_cast<float *>(pk + (kParts - 1) * kRows * kKeep);
        float tau = fminf(fminf(dropped, key_v(keys[kKeep - 1])), tau0);
        epilogue_sync<kEpiWarps>();
        if (group > 0) {
#pragma unroll
            for (int p = 0; p < kKeep; ++p) pk[((group - 1) * kRows + row) * kKeep + p] = keys[p];
            pt[(group - 1) * kRows + row] = tau;
        }
        epilogue_sync<kEpiWarps>();
        if (group == 0) {
#pragma unroll 1
            for (int q = 1; q < kParts; ++q) {
                tau = fminf(tau, pt[(q - 1) * kRows + row]);
#pragma unroll 1
                for (int p = 0; p < kKeep; ++p) {
                    const unsigned long long k = pk[((q - 1) * kRows + row) * kKeep + p];
                    if (k != kNoKey) keep_insert(keys, k, tau);
                }
            }
            if (valid && !*(volatile int *)&S.abort) {
                const int64_t o = static_cast<int64_t>(split) * a.lda + r;
#pragma unroll
                for (int p = 0; p < kKeep; ++p) a.part_key[o * kKeep + p] = keys[p];
                a.part_tau[o] = tau;
            }
        }
    }
    tc_teardown<kEpiWarps>(S, a.status);
}

}  // namespace

bool tc_scan_supported(int dk) { return (dk == 32 || dk == 64) && tensor_maps_available(); }

cudaError_t launch_tc_scan(const ScanArgs &a, const float *Xa_hi, const float *Xa_lo,
                           const float *Xs_hi, const float *Xs_lo, int row_tiles, int splits,
                           cudaStream_t s) {
    TcScanParams P;
    P.a = a;
    P.a_hi = Xa_hi;
    P.a_lo = Xa_lo;
    const int dk_mma = a.f16 ? a.dk / 2 : a.dk;
    if ((a.f16 && dk_mma != kSlab) || !make_point_map(&P.maps.b_hi, Xs_hi, a.ldx, dk_mma) ||
        !make_point_map(&P.maps.b_lo, Xs_lo, a.ldx, dk_mma))
        return cudaErrorInvalidValue;
    const auto kernel = a.f16 ? tc_scan_kernel<true> : tc_scan_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kPipeSmem));
    if (e != cudaSuccess) return e;
    kernel<<<dim3(row_tiles, splits), kScanThreads, kPipeSmem, s>>>(P);
    return cudaGetLastError();
}

cudaError_t tc_scan_test_hooks(unsigned long long wait_ns, int withhold) {
    return tc::set_test_hooks(wait_ns, withhold);
}

}  // namespace hdbmst
