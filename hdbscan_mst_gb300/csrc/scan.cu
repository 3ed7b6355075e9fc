// K6: the Boruvka scan - every active point's cheapest edge to another
// component (page "HDBSCAN", gpu/hdbscan, "Exact shortcuts": only the points
// the shortcuts leave are scanned against all others, over a list of active
// points).
//
// Three kernels, the same scheme as the k-NN search:
//  * mst_scan_kernel ranks every (active row a, point b) pair of different
//    components by an approximate squared weight from the FFMA tile: with
//    t = |b|^2 - 2 a.b (the row's |a|^2 dropped),
//        v = max(t, core_b^2 - |a|^2, core_a^2 - |a|^2)  ~  w(a, b)^2 - |a|^2.
//    Each thread keeps, per row, its best (v, b) and the second-best v; at the
//    end the 16 threads of a row keep the 4 best and a threshold tau that
//    every candidate they dropped reaches or exceeds.
//  * mst_refine_kernel re-evaluates the kept candidates with the library's
//    exact distance and weight max(core_a, core_b, dist), takes the least
//    (w, b), and proves that no dropped point can weigh as little: the
//    expansion's rounding is bounded, so a dropped point's exact weight is at
//    least sqrt((tau + |a|^2 - E)(1 - (d + 3) u)) (1 - u).  Rows it cannot
//    prove go to mst_exact_kernel.
//  * mst_exact_kernel scans the queued rows against every point with the exact
//    weight (the tile pipeline accumulating exact squared distances).
// All three lower the row's candidate key with atomicMin, so the result per
// point is the exact least (w, other end) over the other components.
#include <climits>
#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "tile.cuh"

namespace hdbmst {

namespace {

constexpr int kKeep = 4;  // candidates kept per row and column split

struct ScanSmem {
    TileBuffers T;
    float rna[kBM];   // |a|^2 of each row
    float rra[kBM];   // core_a^2 - |a|^2
    int rcomp[kBM];
};

__global__ void __launch_bounds__(kThreads, 2) mst_scan_kernel(const ScanArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ScanSmem &S = *reinterpret_cast<ScanSmem *>(smem_raw);
    const int tid = threadIdx.x;
    const int ty = tid >> 4, tx = tid & 15;
    const int r0 = blockIdx.x * kBM;
    const int split = blockIdx.y;
    const int ct_begin = split * a.tiles_per_split;
    const int ct_end = min(ct_begin + a.tiles_per_split, a.col_tiles);

    if (tid < kBM) {
        const int r = r0 + tid;
        const bool ok = r < a.na;
        const float na = ok ? a.act_norm[r] : 0.f;
        const float ca = ok ? a.act_core[r] : 0.f;
        S.rna[tid] = na;
        S.rra[tid] = __fsub_rn(__fmul_rn(ca, ca), na);
        S.rcomp[tid] = ok ? a.act_comp[r] : -1;
    }
    __syncthreads();
    // A row tile whose rows all lie in one component skips the column tiles
    // that lie wholly inside that component (columns are grouped by component).
    const bool uniform =
        __syncthreads_and(tid >= kBM || r0 + tid >= a.na || S.rcomp[tid] == S.rcomp[0]);
    int skip_lo = 0, skip_hi = 0;
    if (uniform && a.comp_start) {
        const int C = S.rcomp[0];
        const int c0 = a.comp_start[C], c1 = c0 + a.comp_size[C];
        skip_lo = (c0 + kBN - 1) / kBN;
        skip_hi = c1 / kBN;
    }

    unsigned long long best[8];
    float second[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        best[i] = kNoKey;
        second[i] = INFINITY;
    }
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    if (tid == 0 && a.tile_pairs) {
        const int gap = max(0, min(skip_hi, ct_end) - max(skip_lo, ct_begin));
        atomicAdd(a.tile_pairs,
                  static_cast<unsigned long long>(ct_end - ct_begin - gap) * kBM * kBN);
    }
    tile_pipeline(S.T, a.Xa, a.lda, r0, a.Xs, a.ldx, ct_begin, ct_end, skip_lo, skip_hi, a.dk, acc,
                  [&](float (&ac)[8][8], int ct) {
        const int col0 = ct * kBN;
        float nb[8];
        {
            const float4 v0 = __ldg(reinterpret_cast<const float4 *>(a.col_norm + col0 + tx * 4));
            const float4 v1 = __ldg(reinterpret_cast<const float4 *>(a.col_norm + col0 + 64 + tx * 4));
            nb[0] = v0.x; nb[1] = v0.y; nb[2] = v0.z; nb[3] = v0.w;
            nb[4] = v1.x; nb[5] = v1.y; nb[6] = v1.z; nb[7] = v1.w;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float sig = second[i];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float t = __fmaf_rn(-2.f, ac[i][j], nb[j]);  // +inf past the last point
                ac[i][j] = 0.f;
                if (t < sig) {
                    const int r = row_of(ty, i);
                    const int c = col0 + col_of(tx, j);
                    if (c < a.n && __ldg(a.col_comp + c) != S.rcomp[r]) {
                        const float cb = __ldg(a.col_core + c);
                        const float v = fmaxf(fmaxf(t, __fsub_rn(__fmul_rn(cb, cb), S.rna[r])),
                                              S.rra[r]);
                        const unsigned long long key =
                            (static_cast<unsigned long long>(float_order(v)) << 32) |
                            static_cast<unsigned>(__ldg(a.col_orig + c));
                        if (key < best[i]) {
                            if (best[i] != kNoKey)
                                second[i] = fminf(second[i],
                                                  order_float(static_cast<unsigned>(best[i] >> 32)));
                            best[i] = key;
                        } else if (v < second[i]) {
                            second[i] = v;
                        }
                    }
                }
            }
        }
    });

    // Per row: the 4 best of the 16 threads' bests, and tau = the least value
    // any dropped candidate can have (threads' seconds, and the 5th best).
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        unsigned long long key = best[i];
#pragma unroll
        for (int size = 2; size <= 16; size <<= 1) {
#pragma unroll
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, stride);
                const bool up = (tx & size) == 0;
                const bool lower = (tx & stride) == 0;
                key = (lower == up) ? min(key, other) : max(key, other);
            }
        }
        float tau = second[i];
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) tau = fminf(tau, __shfl_xor_sync(0xffffffffu, tau, o));
        const unsigned long long fifth = __shfl_sync(0xffffffffu, key, (threadIdx.x & 16) + kKeep);
        if (fifth != kNoKey) tau = fminf(tau, order_float(static_cast<unsigned>(fifth >> 32)));
        const int r = r0 + row_of(ty, i);
        if (r < a.na) {
            const int64_t o = static_cast<int64_t>(split) * a.lda + r;
            if (tx < kKeep) a.part_key[o * kKeep + tx] = key;
            if (tx == 0) a.part_tau[o] = tau;
        }
    }
}

// One warp per active row: exact weights of the kept candidates, the least
// key, and the proof that nothing dropped weighs as little.
__global__ void __launch_bounds__(256) mst_refine_kernel(const ScanArgs a) {
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= a.na) return;  // whole warp
    const int g = a.act_idx[r];
    const int q = lane % kKeep;
    const float ca = a.act_core[r];
    // the splits' kept candidates, 32 / kKeep splits per pass of the warp
    unsigned long long exact = kNoKey;
    float tau = INFINITY;
    for (int sb = 0; sb < a.splits; sb += 32 / kKeep) {
        const int s = sb + lane / kKeep;
        const unsigned long long key =
            s < a.splits ? a.part_key[(static_cast<int64_t>(s) * a.lda + r) * kKeep + q] : kNoKey;
        if (key == kNoKey) continue;
        const int b = static_cast<int>(key & 0xffffffffu);
        const float4 *xa = reinterpret_cast<const float4 *>(a.Xp + static_cast<int64_t>(g) * a.dk);
        const float4 *xb = reinterpret_cast<const float4 *>(a.Xp + static_cast<int64_t>(b) * a.dk);
        float acc = 0.f;
        for (int f = 0; f < a.dk / 4; ++f) {
            const float4 u = __ldg(xa + f), v = __ldg(xb + f);
            acc = sqdiff_fma(u.x, v.x, acc);
            acc = sqdiff_fma(u.y, v.y, acc);
            acc = sqdiff_fma(u.z, v.z, acc);
            acc = sqdiff_fma(u.w, v.w, acc);
        }
        const float w = fmaxf(fmaxf(ca, __ldg(a.core + b)), __fsqrt_rn(acc));
        exact = min(exact, key64(w, static_cast<unsigned>(b)));
    }
    for (int s = lane; s < a.splits; s += 32)
        tau = fminf(tau, a.part_tau[static_cast<int64_t>(s) * a.lda + r]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        exact = min(exact, __shfl_xor_sync(0xffffffffu, exact, o));
        tau = fminf(tau, __shfl_xor_sync(0xffffffffu, tau, o));
    }
    if (lane != 0) return;
    // Proof (lane 0).  A dropped point z has v_z >= tau with
    // v = max(t, core_b^2 - |a|^2, core_a^2 - |a|^2).  If core_a^2 - |a|^2 <
    // tau, either core_z^2 - |a|^2 >= tau or t_z >= tau.  With T = w^2 M (w
    // the best exact weight; M covers the exact float32 evaluation,
    // (1 - (d + 3) u), and strict sqrt ordering, 16 u), the first gives
    // core_z > w; for the second the true squared distance is at least
    // |a|^2 + tau - err_coef (|a|^2 + |z|^2) and, by Cauchy-Schwarz, at least
    // (|z| - |a|)^2, so every z exceeds T once
    // |a|^2 + tau - err_coef (|a|^2 + nb_c) > T with nb_c = (|a| + sqrt(T))^2
    // (less the FP16 operands' absolute error part e0 when they ran).
    //
    // With the component bound U_C (a.ub) the row only matters if it has an
    // edge of weight at most U_C (the component already holds an edge of
    // weight U_C).  The proof then runs with w_ref = min(w, U_C): columns the
    // pruned blocks left out have float32 weights above U_C by the pruning
    // bound; if the proof holds and w > U_C, the row has no edge at or below
    // U_C - its kept edge is real but not necessarily its least, so the row
    // is not cached for the next round (act_flag cleared).
    bool proven = false;
    const float uc = a.ub ? __uint_as_float(a.ub[a.act_comp[r]]) : INFINITY;
    const float bw = exact != kNoKey ? key_w(exact) : INFINITY;
    const float wref = fminf(bw, uc);
    if (wref < INFINITY) {
        const float na = a.act_norm[r];
        const float ra = __fsub_rn(__fmul_rn(ca, ca), na);
        const float T = proof_T_up(wref, a.d);
        proven = (ra < tau) && (proof_lhs_down(tau, na, T, a.err_c, *a.e0) > T);
        if (exact != kNoKey) atomicMin(&a.cand[g], exact);
        if (proven && bw > uc && a.act_flag) a.act_flag[g] = 0;
    } else {
        proven = !(tau < INFINITY);  // nothing kept and nothing dropped: no other component
    }
    if (!proven) {
        const int pos = atomicAdd(a.fb_count, 1);
        a.fb_rows[pos] = g;
    }
}

// Queued rows (gathered like the active rows): the exact least (w, other end)
// over all points of other components, on the same tile pipeline but
// accumulating the exact squared distance, so every weight is the library's.
__global__ void __launch_bounds__(kThreads, 2) mst_exact_kernel(const ScanArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ScanSmem &S = *reinterpret_cast<ScanSmem *>(smem_raw);
    const int tid = threadIdx.x;
    const int ty = tid >> 4, tx = tid & 15;
    const int r0 = blockIdx.x * kBM;
    const int ct_begin = blockIdx.y * a.tiles_per_split;
    const int ct_end = min(ct_begin + a.tiles_per_split, a.col_tiles);
    if (tid < kBM) {
        const int r = r0 + tid;
        const bool ok = r < a.na;
        S.rna[tid] = ok ? a.act_core[r] : 0.f;  // core_a
        S.rcomp[tid] = ok ? a.act_comp[r] : -1;
    }
    __syncthreads();
    const bool uniform =
        __syncthreads_and(tid >= kBM || r0 + tid >= a.na || S.rcomp[tid] == S.rcomp[0]);
    int skip_lo = 0, skip_hi = 0;
    if (uniform) {
        const int C = S.rcomp[0];
        const int c0 = a.comp_start[C], c1 = c0 + a.comp_size[C];
        skip_lo = (c0 + kBN - 1) / kBN;
        skip_hi = c1 / kBN;
    }
    unsigned long long best[8];
    float thr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        best[i] = kNoKey;
        thr[i] = INFINITY;
    }
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    tile_pipeline<true>(S.T, a.Xa, a.lda, r0, a.Xs, a.ldx, ct_begin, ct_end, skip_lo, skip_hi,
                        a.dk, acc, [&](float (&ac)[8][8], int ct) {
        const int col0 = ct * kBN;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float d2 = ac[i][j];
                ac[i][j] = 0.f;
                const int c = col0 + col_of(tx, j);
                if (d2 <= thr[i] && c < a.n) {
                    const int r = row_of(ty, i);
                    if (__ldg(a.col_comp + c) != S.rcomp[r]) {
                        const float w = fmaxf(fmaxf(S.rna[r], __ldg(a.col_core + c)),
                                              __fsqrt_rn(d2));
                        const unsigned long long key =
                            key64(w, static_cast<unsigned>(__ldg(a.col_orig + c)));
                        if (key < best[i]) {
                            best[i] = key;
                            // sqrt(d2) <= w requires d2 <= w^2 (1 + 2.1 u): every
                            // pair that could tie or win passes this threshold
                            thr[i] = __fmul_rn(__fmul_rn(w, w), 1.0f + 0x1p-20f);
                        }
                    }
                }
            }
        }
    });
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        unsigned long long k = best[i];
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) k = min(k, __shfl_xor_sync(0xffffffffu, k, o));
        const int r = r0 + row_of(ty, i);
        if (tx == 0 && r < a.na && k != kNoKey) atomicMin(&a.cand[a.act_idx[r]], k);
    }
}

}  // namespace

size_t scan_part_entries(int splits, int64_t lda) {
    return static_cast<size_t>(splits) * lda * kKeep;
}

cudaError_t launch_scan(const ScanArgs &a, int row_tiles, int splits, cudaStream_t s) {
    const size_t smem = sizeof(ScanSmem);
    cudaError_t e = cudaFuncSetAttribute(mst_scan_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    mst_scan_kernel<<<dim3(row_tiles, splits), kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_scan_refine(const ScanArgs &a, cudaStream_t s) {
    mst_refine_kernel<<<(a.na + 7) / 8, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_scan_exact(const ScanArgs &a, int row_tiles, int splits, cudaStream_t s) {
    const size_t smem = sizeof(ScanSmem);
    cudaError_t e = cudaFuncSetAttribute(mst_exact_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    mst_exact_kernel<<<dim3(row_tiles, splits), kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace hdbmst
