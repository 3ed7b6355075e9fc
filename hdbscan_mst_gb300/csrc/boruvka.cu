// K3-K5, K7, K8: Boruvka rounds of the mutual-reachability minimum spanning
// tree (the scan, K6, is in scan.cu).
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
                                unsigned long long *ck64, unsigned *chi, unsigned *ub,
                                unsigned long long *cache) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    comp[i] = i;
    cand[i] = kNoKey;
    cache[i] = kNoKey;
    ck64[i] = kNoKey;
    chi[i] = 0xffffffffu;
    ub[i] = __float_as_uint(INFINITY);
}

// K3: per point, its lightest listed edge into another component (a real
// edge), whether that edge is proven cheapest, and the component bound.
//
// A point also keeps the exact cheapest edge it had in the previous round
// (cache).  Components only grow, so the points outside its component now are
// a subset of those then; if that edge's other end is still outside, it is
// still the cheapest and the point needs no scan.
__global__ void nbr_candidate_kernel(int n, int L, const int32_t *__restrict__ kidx,
                                     const float *__restrict__ kdist,
                                     const float *__restrict__ core, const int *__restrict__ comp,
                                     const unsigned long long *__restrict__ cache,
                                     unsigned long long *__restrict__ cand,
                                     unsigned char *__restrict__ proven,
                                     unsigned *__restrict__ ub, unsigned *__restrict__ status) {
    const int a = blockIdx.x * blockDim.x + threadIdx.x;
    if (a >= n) return;
    const float ca = core[a];
    const int cc = comp[a];
    const unsigned long long held = cache[a];
    if (held != kNoKey && comp[key_i(held)] != cc) {
        cand[a] = held;
        proven[a] = 1;
        atomicMin(&ub[cc], static_cast<unsigned>(held >> 32));
        return;
    }
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

// K5: which points still need a scan (active), and per component the number
// of points and of active points.  Counts are aggregated per warp over lanes
// of the same component.
__global__ void classify_kernel(int n, const unsigned char *__restrict__ proven,
                                const float *__restrict__ core, const int *__restrict__ comp,
                                const unsigned *__restrict__ ub,
                                unsigned char *__restrict__ act_flag, int *__restrict__ size,
                                int *__restrict__ act_size, int *__restrict__ act_count) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31;
    const bool valid = i < n;
    const int c = valid ? comp[i] : -1;
    bool act = valid;
    if (act && proven && proven[i]) act = false;
    // skip only when core_a exceeds the bound strictly: an equal weight could
    // still win on index
    if (act && ub && core[i] > __uint_as_float(ub[c])) act = false;
    if (valid) act_flag[i] = act ? 1 : 0;
    const unsigned peers = __match_any_sync(0xffffffffu, c);
    if (valid && lane == __ffs(peers) - 1) atomicAdd(&size[c], __popc(peers));
    const unsigned actb = __ballot_sync(0xffffffffu, act);
    const unsigned apeers = peers & actb;
    if (act && lane == __ffs(apeers) - 1) atomicAdd(&act_size[c], __popc(apeers));
    if (lane == 0 && actb) atomicAdd(act_count, __popc(actb));
}

// Give every component a contiguous slot range for its points and for its
// active points (slot order between components is arbitrary).
__global__ void slots_kernel(int n, const int *__restrict__ size, const int *__restrict__ act_size,
                             int *__restrict__ start, int *__restrict__ act_start,
                             int *__restrict__ totals) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31;
    const int s = c < n ? size[c] : 0;
    const int a = c < n ? act_size[c] : 0;
    int is = s, ia = a;  // inclusive warp prefix sums
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int ys = __shfl_up_sync(0xffffffffu, is, o);
        const int ya = __shfl_up_sync(0xffffffffu, ia, o);
        if (lane >= o) {
            is += ys;
            ia += ya;
        }
    }
    int bs = 0, ba = 0;
    if (lane == 31) {
        if (is) bs = atomicAdd(&totals[0], is);
        if (ia) ba = atomicAdd(&totals[1], ia);
    }
    bs = __shfl_sync(0xffffffffu, bs, 31);
    ba = __shfl_sync(0xffffffffu, ba, 31);
    if (c < n) {
        start[c] = bs + is - s;
        act_start[c] = ba + ia - a;
    }
}

// Every point to its component's slot range: the column order of the scan
// (perm, and the column arrays in that order) and the active rows grouped by
// component.  Order inside a component is arbitrary; results do not depend
// on it.
__global__ void group_kernel(int n, const int *__restrict__ comp, const float *__restrict__ core,
                             const float *__restrict__ norm,
                             const unsigned char *__restrict__ act_flag,
                             const int *__restrict__ start, const int *__restrict__ act_start,
                             int *__restrict__ cursor, int *__restrict__ act_cursor,
                             int *__restrict__ perm, int *__restrict__ col_comp,
                             float *__restrict__ col_core, float *__restrict__ col_norm,
                             int *__restrict__ act_idx) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31;
    const bool valid = i < n;
    const int c = valid ? comp[i] : -1;
    const bool act = valid && act_flag[i];
    const unsigned peers = __match_any_sync(0xffffffffu, c);
    const int leader = __ffs(peers) - 1;
    int base = 0;
    if (valid && lane == leader) base = atomicAdd(&cursor[c], __popc(peers));
    base = __shfl_sync(0xffffffffu, base, leader);
    const unsigned apeers = peers & __ballot_sync(0xffffffffu, act);
    const int aleader = apeers ? __ffs(apeers) - 1 : 0;
    int abase = 0;
    if (act && lane == aleader) abase = atomicAdd(&act_cursor[c], __popc(apeers));
    abase = __shfl_sync(0xffffffffu, abase, aleader);
    if (valid) {
        const int pos = start[c] + base + __popc(peers & lanemask_lt());
        perm[pos] = i;
        col_comp[pos] = c;
        col_core[pos] = core[i];
        col_norm[pos] = norm[i];
    }
    if (act) act_idx[act_start[c] + abase + __popc(apeers & lanemask_lt())] = i;
}

// Columns in grouped order into their own feature-major buffer; padding
// columns are zero.
__global__ void gather_cols_kernel(int n, int n_pad, const int *__restrict__ perm,
                                   const float *__restrict__ Xf, float *__restrict__ Xs) {
    const int pos = blockIdx.x * blockDim.x + threadIdx.x;
    const int f = blockIdx.y;
    if (pos >= n_pad) return;
    const int g = pos < n ? perm[pos] : -1;
    Xs[static_cast<int64_t>(f) * n_pad + pos] = g >= 0 ? Xf[static_cast<int64_t>(f) * n_pad + g] : 0.f;
}

// Padding columns of the grouped order never rank (+inf norm).
__global__ void pad_norms_kernel(int n, int n_pad, float *__restrict__ col_norm) {
    const int pos = n + blockIdx.x * blockDim.x + threadIdx.x;
    if (pos < n_pad) col_norm[pos] = INFINITY;
}

// Point-major rows by index, hi and lo parts, one float4 per thread.
__global__ void gather_points_kernel(int count, int count_pad, int dk, const int *__restrict__ idx,
                                     const float4 *__restrict__ src_hi,
                                     const float4 *__restrict__ src_lo, float4 *__restrict__ dst_hi,
                                     float4 *__restrict__ dst_lo) {
    const int q4 = dk / 4;
    const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= static_cast<int64_t>(count_pad) * q4) return;
    const int r = static_cast<int>(e / q4), q = static_cast<int>(e - static_cast<int64_t>(r) * q4);
    float4 h = make_float4(0.f, 0.f, 0.f, 0.f), l = h;
    if (r < count) {
        const int64_t g = static_cast<int64_t>(idx[r]) * q4 + q;
        h = src_hi[g];
        l = src_lo[g];
    }
    dst_hi[e] = h;
    dst_lo[e] = l;
}

// Active rows into their own padded feature-major buffer (skipped when Xa is
// null), with their core distance, component and squared norm.
__global__ void gather_kernel(int na, int na_pad, int dk, const int *__restrict__ act_idx,
                              const float *__restrict__ Xf, int64_t ldx,
                              const float *__restrict__ core, const int *__restrict__ comp,
                              const float *__restrict__ norm, float *__restrict__ Xa,
                              float *__restrict__ act_core, int *__restrict__ act_comp,
                              float *__restrict__ act_norm) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    const int f = blockIdx.y;
    if (r >= na_pad) return;
    const int g = r < na ? act_idx[r] : -1;
    if (Xa)
        Xa[static_cast<int64_t>(f) * na_pad + r] = g >= 0 ? Xf[static_cast<int64_t>(f) * ldx + g] : 0.f;
    if (f == 0) {
        act_core[r] = g >= 0 ? core[g] : 0.f;
        act_comp[r] = g >= 0 ? comp[g] : -1;
        act_norm[r] = g >= 0 ? norm[g] : 0.f;
    }
}

// K7: per component, the least (w, lo, hi) over its points' candidates, in
// two stages of 32-bit words: (w, lo) as one 64-bit key, then hi among the
// candidates that hold the least (w, lo).  Each stage first reduces within
// the warp over the lanes of the same component (__match_any_sync groups
// them; __reduce_min_sync takes the least w, then the least lo at that w),
// so one lane per component and warp updates global memory.  The first pass
// also records, for the next round, the candidates that are exact (proven,
// or scanned one-sided: act_flag); the others (skipped by the bound, or only
// bounded by the symmetric scan) are not.
__global__ void comp_min_lo_kernel(int n, const unsigned long long *__restrict__ cand,
                                   const int *__restrict__ comp,
                                   unsigned long long *__restrict__ ck64,
                                   const unsigned char *__restrict__ proven,
                                   const unsigned char *__restrict__ act_flag,
                                   unsigned long long *__restrict__ cache) {
    const int a = blockIdx.x * blockDim.x + threadIdx.x;
    const bool in = a < n;
    const unsigned long long k = in ? cand[a] : kNoKey;
    if (in && cache) cache[a] = (proven[a] || (act_flag && act_flag[a])) ? k : kNoKey;
    const bool has = k != kNoKey;
    const int c = has ? comp[a] : -1;  // lanes without a candidate form their own group
    const unsigned wb = has ? static_cast<unsigned>(k >> 32) : 0xffffffffu;
    const unsigned lo = has ? min(static_cast<unsigned>(a), key_i(k)) : 0xffffffffu;
    const unsigned peers = __match_any_sync(0xffffffffu, c);
    const unsigned wmin = __reduce_min_sync(peers, wb);
    const unsigned lomin = __reduce_min_sync(peers, wb == wmin ? lo : 0xffffffffu);
    if (has && (threadIdx.x & 31) == __ffs(peers) - 1)
        atomicMin(&ck64[c], (static_cast<unsigned long long>(wmin) << 32) | lomin);
}

__global__ void comp_min_hi_kernel(int n, const unsigned long long *__restrict__ cand,
                                   const int *__restrict__ comp,
                                   const unsigned long long *__restrict__ ck64,
                                   unsigned *__restrict__ chi) {
    const int a = blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned long long k = a < n ? cand[a] : kNoKey;
    int c = -1;
    unsigned hi = 0xffffffffu;
    if (k != kNoKey) {
        const unsigned b = key_i(k);
        const unsigned lo = min(static_cast<unsigned>(a), b);
        const int ca = comp[a];
        if (((k & 0xffffffff00000000ull) | lo) == ck64[ca]) {
            c = ca;
            hi = max(static_cast<unsigned>(a), b);
        }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, c);
    const unsigned himin = __reduce_min_sync(peers, hi);
    if (c >= 0 && (threadIdx.x & 31) == __ffs(peers) - 1) atomicMin(&chi[c], himin);
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

// Root of every component by pointer jumping, in a counter-bounded number of
// launches (the merge of page "HDBSCAN", "The algorithm on the device", on
// the device).  The hooks form a forest over the components; its depth is
// below the number of components.  The first launch walks each component's
// parent pointers for at most kJumpSteps steps; every further launch walks
// at most kJumpSteps steps over the pointers the launches before it wrote,
// each of which already skips kJumpSteps^j levels (or ends at a root), so
// after launch j every pointer is kJumpSteps^(j+1) levels up or at its
// root.  root_of[x] == x exactly for the roots.  Updates happen in place:
// a pointer read while another thread rewrites it is still an ancestor, so
// a fresher value only helps.  A launch returns at once when the launch
// before it found every pointer at a root (live[j] holds the round stamp of
// the last launch j that did not); relabel_kernel checks the result.
constexpr int kJumpSteps = 16;

__global__ void roots_init_kernel(int n, const int *__restrict__ comp,
                                  const int *__restrict__ parent, int *__restrict__ root_of,
                                  int *__restrict__ live, int stamp) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= n || comp[c] != c) return;
    int r = c;
#pragma unroll 1
    for (int s = 0; s < kJumpSteps; ++s) {
        const int p = parent[r];
        if (p == r) break;
        r = p;
    }
    root_of[c] = r;
    if (parent[r] != r) live[0] = stamp;
}

__global__ void roots_jump_kernel(int n, const int *__restrict__ comp, int *root_of, int *live,
                                  int pass, int stamp) {
    if (live[pass - 1] != stamp) return;  // every pointer already at its root
    for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < n; c += gridDim.x * blockDim.x) {
        if (comp[c] != c) continue;
        int r = root_of[c];
#pragma unroll 1
        for (int s = 0; s < kJumpSteps; ++s) {
            const int p = root_of[r];
            if (p == r) break;
            r = p;
        }
        root_of[c] = r;
        if (root_of[r] != r) live[pass] = stamp;
    }
}

// Every point takes its component's root; a root that is not one (the
// bounded jumping did not reach it) is reported instead of used.
__global__ void relabel_kernel(int n, int *__restrict__ comp, const int *__restrict__ root_of,
                               const int *__restrict__ parent,
                               unsigned long long *__restrict__ cand,
                               unsigned long long *__restrict__ ck64, unsigned *__restrict__ chi,
                               unsigned *__restrict__ ub, unsigned *__restrict__ status) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int r = root_of[comp[i]];
    if (parent[r] != r) atomicOr(status, kStatusNoConverge);
    comp[i] = r;
    cand[i] = kNoKey;
    ck64[i] = kNoKey;
    chi[i] = 0xffffffffu;
    ub[i] = __float_as_uint(INFINITY);
}

inline int blocks_for(int n, int t) { return (n + t - 1) / t; }

}  // namespace

cudaError_t launch_mst_init(int n, int *comp, unsigned long long *cand, unsigned long long *ck64,
                            unsigned *chi, unsigned *ub, unsigned long long *cache,
                            cudaStream_t s) {
    mst_init_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, comp, cand, ck64, chi, ub, cache);
    return cudaGetLastError();
}

cudaError_t launch_nbr_candidate(int n, int L, const int32_t *kidx, const float *kdist,
                                 const float *core, const int *comp,
                                 const unsigned long long *cache, unsigned long long *cand,
                                 unsigned char *proven, unsigned *ub, unsigned *status,
                                 cudaStream_t s) {
    nbr_candidate_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, L, kidx, kdist, core, comp, cache,
                                                            cand, proven, ub, status);
    return cudaGetLastError();
}

cudaError_t launch_classify(int n, const unsigned char *proven, const float *core,
                            const int *comp, const unsigned *ub, unsigned char *act_flag,
                            int *size, int *act_size, int *act_count, cudaStream_t s) {
    classify_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, proven, core, comp, ub, act_flag, size,
                                                       act_size, act_count);
    return cudaGetLastError();
}

cudaError_t launch_group(int n, int n_pad, const int *comp, const float *core, const float *norm,
                         const unsigned char *act_flag, const int *size, const int *act_size,
                         int *start, int *act_start, int *cursor, int *act_cursor, int *totals,
                         int *perm, int *col_comp, float *col_core, float *col_norm, int *act_idx,
                         cudaStream_t s) {
    slots_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, size, act_size, start, act_start, totals);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    group_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, comp, core, norm, act_flag, start, act_start,
                                                    cursor, act_cursor, perm, col_comp, col_core,
                                                    col_norm, act_idx);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_extra_launches(1);
    if (n_pad > n) {
        pad_norms_kernel<<<blocks_for(n_pad - n, 256), 256, 0, s>>>(n, n_pad, col_norm);
        count_extra_launches(1);
    }
    return cudaGetLastError();
}

cudaError_t launch_gather_cols(int n, int n_pad, int dk, const int *perm, const float *Xf,
                               float *Xs, cudaStream_t s) {
    gather_cols_kernel<<<dim3(blocks_for(n_pad, 256), dk), 256, 0, s>>>(n, n_pad, perm, Xf, Xs);
    return cudaGetLastError();
}

cudaError_t launch_gather_points(int count, int count_pad, int dk, const int *idx,
                                 const float *src_hi, const float *src_lo, float *dst_hi,
                                 float *dst_lo, cudaStream_t s) {
    const int64_t total = static_cast<int64_t>(count_pad) * (dk / 4);
    gather_points_kernel<<<static_cast<int>((total + 255) / 256), 256, 0, s>>>(
        count, count_pad, dk, idx, reinterpret_cast<const float4 *>(src_hi),
        reinterpret_cast<const float4 *>(src_lo), reinterpret_cast<float4 *>(dst_hi),
        reinterpret_cast<float4 *>(dst_lo));
    return cudaGetLastError();
}

cudaError_t launch_gather(int na, int na_pad, int dk, const int *act_idx, const float *Xf,
                          int64_t ldx, const float *core, const int *comp, const float *norm,
                          float *Xa, float *act_core, int *act_comp, float *act_norm,
                          cudaStream_t s) {
    gather_kernel<<<dim3(blocks_for(na_pad, 256), Xa ? dk : 1), 256, 0, s>>>(
        na, na_pad, dk, act_idx, Xf, ldx, core, comp, norm, Xa, act_core, act_comp, act_norm);
    return cudaGetLastError();
}

cudaError_t launch_comp_min(int n, const unsigned long long *cand, const int *comp,
                            unsigned long long *ck64, unsigned *chi, const unsigned char *proven,
                            const unsigned char *act_flag, unsigned long long *cache,
                            cudaStream_t s, int stage) {
    if (stage == 0)
        comp_min_lo_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, cand, comp, ck64, proven,
                                                              act_flag, cache);
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

int roots_launches(int components) {
    int launches = 1;
    int64_t reach = kJumpSteps;
    while (reach < components && launches < kJumpMaxLaunches) {
        reach *= kJumpSteps;
        ++launches;
    }
    return launches;
}

cudaError_t launch_roots(int n, int components, const int *comp, const int *parent, int *root_of,
                         int *live, int stamp, int sms, cudaStream_t s, int launch_cap) {
    roots_init_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, comp, parent, root_of, live, stamp);
    cudaError_t e = cudaGetLastError();
    int launches = roots_launches(components);
    if (launch_cap > 0) launches = std::min(launches, launch_cap);
    const int grid = std::max(1, std::min(blocks_for(n, 256), 4 * sms));
    for (int j = 1; j < launches && e == cudaSuccess; ++j) {
        roots_jump_kernel<<<grid, 256, 0, s>>>(n, comp, root_of, live, j, stamp);
        count_extra_launches(1);
        e = cudaGetLastError();
    }
    return e;
}

cudaError_t launch_relabel(int n, int *comp, const int *root_of, const int *parent,
                           unsigned long long *cand, unsigned long long *ck64, unsigned *chi,
                           unsigned *ub, unsigned *status, cudaStream_t s) {
    relabel_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, comp, root_of, parent, cand, ck64, chi,
                                                      ub, status);
    return cudaGetLastError();
}

}  // namespace hdbmst
