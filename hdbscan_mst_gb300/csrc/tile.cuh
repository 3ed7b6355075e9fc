// The register-blocked FFMA distance tile shared by the k-NN search and the
// Boruvka scan.
//
// A CTA of 256 threads owns 128 rows x 128 columns; thread (ty, tx) holds an
// 8 x 8 block of dot products acc[i][j] = x_row . y_col for rows
// row_of(ty, i) and columns col_of(tx, j) (two 4-wide halves 64 apart, so a
// warp's float4 shared loads are conflict-free).  Features stream through
// shared memory in chunks of kBK with cp.async double buffering; the column
// tiles of a CTA's range follow one another in the same pipeline, and after
// the last chunk of each column tile the caller's epilogue consumes acc.
#pragma once

#include "common.cuh"

namespace hdbmst {

struct TileBuffers {
    float As[2][kBK][kBM];
    float Bs[2][kBK][kBN];
};

__device__ __forceinline__ int row_of(int ty, int i) { return (i < 4 ? 0 : 60) + ty * 4 + i; }
__device__ __forceinline__ int col_of(int tx, int j) { return (j < 4 ? 0 : 60) + tx * 4 + j; }

// Runs the pipeline over column tiles [ct_begin, ct_end) of B against the 128
// rows of A starting at column r0 (A and B feature-major, dk features, padded
// so every row tile and column tile is whole).  epi(acc, ct) is called once
// per column tile with the finished dot products; it must leave acc zeroed.
//
// Column tiles in [skip_lo, skip_hi) are left out (an empty interval skips
// nothing); the Boruvka scan uses it to pass over a row tile's own component.
//
// kDiff = false accumulates dot products (one FFMA per feature); kDiff = true
// accumulates the library's exact squared distance instead (difference, then
// fused square-add, features in ascending order).
template <bool kDiff = false, class Epilogue>
__device__ __forceinline__ void tile_pipeline(TileBuffers &T, const float *__restrict__ A,
                                              int64_t lda, int r0, const float *__restrict__ B,
                                              int64_t ldb, int ct_begin, int ct_end, int skip_lo,
                                              int skip_hi, int dk, float (&acc)[8][8],
                                              Epilogue &&epi) {
    const int tid = threadIdx.x;
    const int ty = tid >> 4, tx = tid & 15;
    const int nchunks = dk / kBK;
    const int s_lo = min(max(skip_lo, ct_begin), ct_end);
    const int s_hi = max(min(skip_hi, ct_end), s_lo);
    const int gap = s_hi - s_lo;
    const int nsteps = max(ct_end - ct_begin - gap, 0) * nchunks;
    auto tile_at = [&](int k) {
        const int t = ct_begin + k;
        return t >= s_lo ? t + gap : t;
    };

    auto issue = [&](int step, int buf) {
        const int ct = tile_at(step / nchunks);
        const int kc = step - (step / nchunks) * nchunks;
        const float *ga = A + static_cast<int64_t>(kc * kBK) * lda + r0;
        const float *gb = B + static_cast<int64_t>(kc * kBK) * ldb + static_cast<int64_t>(ct) * kBN;
#pragma unroll
        for (int v = tid; v < kBK * kBM / 4; v += kThreads) {
            const int kr = v >> 5, c4 = (v & 31) * 4;
            cp_async16(&T.As[buf][kr][c4], ga + static_cast<int64_t>(kr) * lda + c4);
            cp_async16(&T.Bs[buf][kr][c4], gb + static_cast<int64_t>(kr) * ldb + c4);
        }
        cp_async_commit();
    };

    if (nsteps > 0) issue(0, 0);
    for (int step = 0; step < nsteps; ++step) {
        const int buf = step & 1;
        cp_async_wait_all();
        __syncthreads();
        if (step + 1 < nsteps) issue(step + 1, buf ^ 1);
#pragma unroll
        for (int kk = 0; kk < kBK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&T.As[buf][kk][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&T.As[buf][kk][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&T.Bs[buf][kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&T.Bs[buf][kk][64 + tx * 4]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    acc[i][j] = kDiff ? sqdiff_fma(av[i], bv[j], acc[i][j])
                                      : __fmaf_rn(av[i], bv[j], acc[i][j]);
        }
        if ((step + 1) % nchunks == 0) epi(acc, tile_at(step / nchunks));
    }
}


}  // namespace hdbmst
