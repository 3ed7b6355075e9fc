// K3-K8: Boruvka rounds of the mutual-reachability minimum spanning tree.
//
// Page "HDBSCAN" (neuro-kitchen dsp-kitchen gpu/hdbscan):
//  * "The algorithm on the device": w(a, b) = max(core_a, core_b, |a - b|);
//    each round every component takes its cheapest edge to another component
//    and components merge along those edges; ties by (weight, lower index,
//    higher index) make the tree unique.
//  * "Exact shortcuts": a point's weight to anything is at least its own core
//    distance.  If its nearest list provably holds every point within that
//    distance (one neighbour more than min_samples, the last strictly farther)
//    and a listed neighbour in another component has a core distance no
//    larger, that edge is the point's cheapest (lowest index on ties).  Every
//    listed edge into another component is a real edge, so the lightest bounds
//    the component's cheapest edge; a point whose core distance exceeds that
//    bound cannot improve it.  Only the remaining points are scanned against
//    all others, over a list of active points.
//
// Keys.  For a fixed point a, ordering its edges by (w, lower, higher) is the
// same as ordering by (w, other endpoint): the other ends below a come first,
// in index order, then those above a.  So a per-point key is the 64-bit
// (w bits, other end).  Per component the full (w, lo, hi) key is 96 bits; it
// is reduced in two passes, a 64-bit atomicMin over (w, lo), then a 32-bit
// atomicMin over hi among the points that match the winning (w, lo).
#include <climits>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace hdbmst {

namespace {

__global__ void mst_init_kernel(int n, int *comp, unsigned long long *cand,
                                unsigned long long *ck64, unsigned *chi, unsigned *ub) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    comp[i] = i;
    cand[i] = kNoKey;
    ck64[i] = kNoKey;
    chi[i] = 0xffffffffu;
    ub[i] = __float_as_uint(INFINITY);
}

// K3: per point, its lightest listed edge into another component (a real
// edge), whether that edge is proven cheapest, and the component bound.
__global__ void nbr_candidate_kernel(int n, int L, const int32_t *__restrict__ kidx,
                                     const float *__restrict__ kdist,
                                     const float *__restrict__ core, const int *__restrict__ comp,
                                     unsigned long long *__restrict__ cand,
                                     unsigned char *__restrict__ proven,
                                     unsigned *__restrict__ ub, unsigned *__restrict__ status) {
    const int a = blockIdx.x * blockDim.x + threadIdx.x;
    if (a >= n) return;
    const float ca = core[a];
    const int cc = comp[a];
    unsigned long long best = kNoKey;
    const int64_t o = static_cast<int64_t>(a) * L;
    for (int l = 0; l < L; ++l) {
        const int b = kidx[o + l];
        if (b < 0 || b >= n) {  // not a list this library wrote: refuse it
            atomicOr(status, kStatusBadList);
            continue;
        }
        if (comp[b] == cc) continue;
        const float w = fmaxf(fmaxf(ca, core[b]), kdist[o + l]);
        best = min(best, key64(w, static_cast<unsigned>(b)));
    }
    // The list holds every point within distance core_a when its last entry
    // lies strictly farther (ties at the edge could hide a lower index).
    const bool complete = kdist[o + L - 1] > ca;
    cand[a] = best;
    proven[a] = (complete && best != kNoKey && key_w(best) == ca) ? 1 : 0;
    if (best != kNoKey) atomicMin(&ub[cc], static_cast<unsigned>(best >> 32));
}

// K5: the points that still need a scan, appended with one atomic per warp.
__global__ void active_kernel(int n, const unsigned char *__restrict__ proven,
                              const float *__restrict__ core, const int *__restrict__ comp,
                              const unsigned *__restrict__ ub, int *__restrict__ act_idx,
                              int *__restrict__ act_count) {
    const int a = blockIdx.x * blockDim.x + threadIdx.x;
    bool act = false;
    if (a < n) {
        act = true;
        if (proven && proven[a]) act = false;
        // skip only when core_a exceeds the bound strictly: an equal weight
        // could still win on index
        if (act && ub && core[a] > __uint_as_float(ub[comp[a]])) act = false;
    }
    const unsigned m = __ballot_sync(0xffffffffu, act);
    int base = 0;
    if ((threadIdx.x & 31) == 0 && m) base = atomicAdd(act_count, __popc(m));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (act) act_idx[base + __popc(m & lanemask_lt())] = a;
}

// Active rows into their own padded feature-major buffer.
__global__ void gather_kernel(int na, int na_pad, int dk, const int *__restrict__ act_idx,
                              const float *__restrict__ Xf, int64_t ldx,
                              const float *__restrict__ core, const int *__restrict__ comp,
                              float *__restrict__ Xa, float *__restrict__ act_core,
                              int *__restrict__ act_comp) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    const int f = blockIdx.y;
    if (r >= na_pad) return;
    const int g = r < na ? act_idx[r] : -1;
    Xa[static_cast<int64_t>(f) * na_pad + r] = g >= 0 ? Xf[static_cast<int64_t>(f) * ldx + g] : 0.f;
    if (f == 0) {
        act_core[r] = g >= 0 ? core[g] : 0.f;
        act_comp[r] = g >= 0 ? comp[g] : -1;
    }
}

// K6: for every active row, the least (w, other end) over all points of other
// components.  Register-blocked 128 x 128 tile like the k-NN engine, but each
// pair accumulates the library's exact squared distance (difference, then
// fused square-add, ascending features), so the weight is bit-identical to
// the one the neighbour lists carry.
struct ScanSmem {
    float As[2][kBK][kBM];
    float Bs[2][kBK][kBN];
    float rcore[kBM];
    int rcomp[kBM];
};

__device__ __forceinline__ int srow(int ty, int i) { return (i < 4 ? 0 : 60) + ty * 4 + i; }
__device__ __forceinline__ int scol(int tx, int j) { return (j < 4 ? 0 : 60) + tx * 4 + j; }

__global__ void __launch_bounds__(kThreads, 2) scan_kernel(const ScanArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ScanSmem &S = *reinterpret_cast<ScanSmem *>(smem_raw);
    const int tid = threadIdx.x;
    const int ty = tid >> 4, tx = tid & 15;
    const int r0 = blockIdx.x * kBM;
    const int ct_begin = blockIdx.y * a.tiles_per_split;
    const int ct_end = min(ct_begin + a.tiles_per_split, a.col_tiles);

    if (tid < kBM) {
        const int r = r0 + tid;
        S.rcore[tid] = r < a.na ? a.act_core[r] : 0.f;
        S.rcomp[tid] = r < a.na ? a.act_comp[r] : -1;
    }
    __syncthreads();

    unsigned long long best[8];
    float thr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        best[i] = kNoKey;
        thr[i] = INFINITY;
    }

    const int nchunks = a.dk / kBK;
    const int nsteps = max(ct_end - ct_begin, 0) * nchunks;
    auto issue = [&](int step, int buf) {
        const int ct = ct_begin + step / nchunks;
        const int kc = step - (step / nchunks) * nchunks;
        const float *ga = a.Xa + static_cast<int64_t>(kc * kBK) * a.lda + r0;
        const float *gb = a.Xf + static_cast<int64_t>(kc * kBK) * a.ldx + static_cast<int64_t>(ct) * kBN;
#pragma unroll
        for (int v = tid; v < kBK * kBM / 4; v += kThreads) {
            const int kr = v >> 5, c4 = (v & 31) * 4;
            cp_async16(&S.As[buf][kr][c4], ga + static_cast<int64_t>(kr) * a.lda + c4);
            cp_async16(&S.Bs[buf][kr][c4], gb + static_cast<int64_t>(kr) * a.ldx + c4);
        }
        cp_async_commit();
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    if (nsteps > 0) issue(0, 0);
    for (int step = 0; step < nsteps; ++step) {
        const int buf = step & 1;
        cp_async_wait_all();
        __syncthreads();
        if (step + 1 < nsteps) issue(step + 1, buf ^ 1);
#pragma unroll
        for (int kk = 0; kk < kBK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&S.As[buf][kk][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&S.As[buf][kk][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&S.Bs[buf][kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&S.Bs[buf][kk][64 + tx * 4]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = sqdiff_fma(av[i], bv[j], acc[i][j]);
        }
        if ((step + 1) % nchunks == 0) {
            const int col0 = (ct_begin + step / nchunks) * kBN;
            float cb[8];
            int cc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int c = col0 + scol(tx, j);
                const bool ok = c < a.n;
                cb[j] = ok ? __ldg(a.core + c) : 0.f;
                cc[j] = ok ? __ldg(a.comp + c) : INT_MIN;  // padding: never another component
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = srow(ty, i);
                const int rc = S.rcomp[r];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float d2 = acc[i][j];
                    if (cc[j] != rc && cc[j] != INT_MIN && d2 <= thr[i]) {
                        const float w = fmaxf(fmaxf(S.rcore[r], cb[j]), __fsqrt_rn(d2));
                        const unsigned long long key =
                            key64(w, static_cast<unsigned>(col0 + scol(tx, j)));
                        if (key < best[i]) {
                            best[i] = key;
                            // sqrt(d2) <= w requires d2 <= w^2 (1 + 2.1 u); this
                            // threshold keeps every pair that could tie or win
                            thr[i] = __fmul_rn(__fmul_rn(w, w), 1.0f + 0x1p-20f);
                        }
                    }
                    acc[i][j] = 0.f;
                }
            }
        }
    }
    // least key per row: the 16 lanes of a half-warp share the same rows
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        unsigned long long k = best[i];
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) k = min(k, __shfl_xor_sync(0xffffffffu, k, o));
        best[i] = k;
    }
    if (tx == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = r0 + srow(ty, i);
            if (r < a.na && best[i] != kNoKey) {
                const int g = a.act_idx ? a.act_idx[r] : r;
                atomicMin(&a.cand[g], best[i]);
            }
        }
    }
}

// K7: per component, the least (w, lo, hi) over its points' candidates.
__global__ void comp_min_lo_kernel(int n, const unsigned long long *__restrict__ cand,
                                   const int *__restrict__ comp,
                                   unsigned long long *__restrict__ ck64) {
    const int a = blockIdx.x * blockDim.x + threadIdx.x;
    if (a >= n) return;
    const unsigned long long k = cand[a];
    if (k == kNoKey) return;
    const unsigned b = key_i(k);
    const unsigned lo = min(static_cast<unsigned>(a), b);
    atomicMin(&ck64[comp[a]], (k & 0xffffffff00000000ull) | lo);
}

__global__ void comp_min_hi_kernel(int n, const unsigned long long *__restrict__ cand,
                                   const int *__restrict__ comp,
                                   const unsigned long long *__restrict__ ck64,
                                   unsigned *__restrict__ chi) {
    const int a = blockIdx.x * blockDim.x + threadIdx.x;
    if (a >= n) return;
    const unsigned long long k = cand[a];
    if (k == kNoKey) return;
    const unsigned b = key_i(k);
    const unsigned lo = min(static_cast<unsigned>(a), b);
    const unsigned hi = max(static_cast<unsigned>(a), b);
    const int c = comp[a];
    if (((k & 0xffffffff00000000ull) | lo) == ck64[c]) atomicMin(&chi[c], hi);
}

// K8: every component hooks onto the component at the other end of its
// cheapest edge.  With one strict order on edges the only cycles among the
// hooks are pairs that chose the same edge; the lower component id stays a
// root there and the edge is recorded once.
__global__ void hook_kernel(int n, const int *__restrict__ comp,
                            const unsigned long long *__restrict__ ck64,
                            const unsigned *__restrict__ chi, int *__restrict__ parent,
                            int *__restrict__ e_lo, int *__restrict__ e_hi,
                            float *__restrict__ e_w, int *__restrict__ edge_count,
                            unsigned *__restrict__ status) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= n || comp[c] != c) return;
    const unsigned long long k = ck64[c];
    if (k == kNoKey) {
        parent[c] = c;
        return;
    }
    const int lo = static_cast<int>(k & 0xffffffffu);
    const int hi = static_cast<int>(chi[c]);
    const int other = comp[lo] == c ? hi : lo;
    const int dc = comp[other];
    const bool mutual = ck64[dc] == k && chi[dc] == static_cast<unsigned>(hi);
    if (mutual && c < dc) {
        parent[c] = c;
        return;
    }
    parent[c] = dc;
    const int pos = atomicAdd(edge_count, 1);
    if (pos < n - 1) {
        e_lo[pos] = lo;
        e_hi[pos] = hi;
        e_w[pos] = key_w(k);
    } else {
        atomicOr(status, kStatusOverflow);
    }
}

// Root of every component: follow parent pointers (read only here), at most
// n steps.
__global__ void roots_kernel(int n, const int *__restrict__ comp, const int *__restrict__ parent,
                             int *__restrict__ root_of, unsigned *__restrict__ status) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= n || comp[c] != c) return;
    int r = c;
    for (int s = 0; s < n; ++s) {
        const int p = parent[r];
        if (p == r) break;
        r = p;
    }
    if (parent[r] != r) atomicOr(status, kStatusNoConverge);
    root_of[c] = r;
}

__global__ void relabel_kernel(int n, int *__restrict__ comp, const int *__restrict__ root_of,
                               unsigned long long *__restrict__ cand,
                               unsigned long long *__restrict__ ck64, unsigned *__restrict__ chi,
                               unsigned *__restrict__ ub) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    comp[i] = root_of[comp[i]];
    cand[i] = kNoKey;
    ck64[i] = kNoKey;
    chi[i] = 0xffffffffu;
    ub[i] = __float_as_uint(INFINITY);
}

inline int blocks_for(int n, int t) { return (n + t - 1) / t; }

}  // namespace

cudaError_t launch_mst_init(int n, int *comp, unsigned long long *cand, unsigned long long *ck64,
                            unsigned *chi, unsigned *ub, cudaStream_t s) {
    mst_init_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, comp, cand, ck64, chi, ub);
    return cudaGetLastError();
}

cudaError_t launch_nbr_candidate(int n, int L, const int32_t *kidx, const float *kdist,
                                 const float *core, const int *comp, unsigned long long *cand,
                                 unsigned char *proven, unsigned *ub, unsigned *status,
                                 cudaStream_t s) {
    nbr_candidate_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, L, kidx, kdist, core, comp, cand,
                                                            proven, ub, status);
    return cudaGetLastError();
}

cudaError_t launch_active(int n, const unsigned char *proven, const float *core, const int *comp,
                          const unsigned *ub, int *act_idx, int *act_count, cudaStream_t s) {
    active_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, proven, core, comp, ub, act_idx,
                                                     act_count);
    return cudaGetLastError();
}

cudaError_t launch_gather(int na, int na_pad, int dk, const int *act_idx, const float *Xf,
                          int64_t ldx, const float *core, const int *comp, float *Xa,
                          float *act_core, int *act_comp, cudaStream_t s) {
    gather_kernel<<<dim3(blocks_for(na_pad, 256), dk), 256, 0, s>>>(
        na, na_pad, dk, act_idx, Xf, ldx, core, comp, Xa, act_core, act_comp);
    return cudaGetLastError();
}

cudaError_t launch_scan(const ScanArgs &a, int row_tiles, int splits, cudaStream_t s) {
    const size_t smem = sizeof(ScanSmem);
    cudaError_t e = cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    scan_kernel<<<dim3(row_tiles, splits), kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_comp_min(int n, const unsigned long long *cand, const int *comp,
                            unsigned long long *ck64, unsigned *chi, cudaStream_t s, int stage) {
    if (stage == 0)
        comp_min_lo_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, cand, comp, ck64);
    else
        comp_min_hi_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, cand, comp, ck64, chi);
    return cudaGetLastError();
}

cudaError_t launch_hook(int n, const int *comp, const unsigned long long *ck64,
                        const unsigned *chi, int *parent, int *e_lo, int *e_hi, float *e_w,
                        int *edge_count, unsigned *status, cudaStream_t s) {
    hook_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, comp, ck64, chi, parent, e_lo, e_hi, e_w,
                                                   edge_count, status);
    return cudaGetLastError();
}

cudaError_t launch_roots(int n, const int *comp, const int *parent, int *root_of,
                         unsigned *status, cudaStream_t s) {
    roots_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, comp, parent, root_of, status);
    return cudaGetLastError();
}

cudaError_t launch_relabel(int n, int *comp, const int *root_of, unsigned long long *cand,
                           unsigned long long *ck64, unsigned *chi, unsigned *ub,
                           cudaStream_t s) {
    relabel_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, comp, root_of, cand, ck64, chi, ub);
    return cudaGetLastError();
}

}  // namespace hdbmst
