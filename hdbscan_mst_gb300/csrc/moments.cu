// The split-product second moment and covariance (page "Covariance",
// gpu/covariance): C = (X - mu)(X - mu)^T / n and X X^T / n over a window of
// n samples [t0, t0 + n) of a channel-major recording, in splits of 4 096
// samples.
//
//  1. stats: one block per channel sums the window in a fixed order
//     (two compensated float32 sums per thread, then float64), giving the channel
//     sum, the mean as a float32 pair (mu_hi + mu_lo), and the channel's
//     scale exponent from its largest |x| and |mu|.
//  2. split: copies the window into a split-major buffer [S][C_pad][4096]
//     (the page's split_rows copy: the batch is the outermost stride, the
//     window's column offset is applied here, so any start column and any
//     odd length are fine, and the last split's tail and the padding
//     channels are zero, which adds nothing to the products).  The centred
//     value v = (x - mu_hi) - mu_lo, for the second moment too, is split into
//     the two-part FP16 operands of the tensor cores: with a power of two 2^e
//     per channel putting the channel's largest magnitude below 2^15,
//     hi = fp16(v 2^e), lo = fp16(v 2^e - hi) (a quiet channel beside a loud
//     one keeps its precision).  Centring keeps the split
//     sums from growing along a split: measured on uncentred windows with a
//     DC level, products of raw values came out 3e-5 off relative to
//     sum |x_i x_j|, centred ones 2e-7.
//  3. product: one CTA per (tile pair I <= J of 128 channels, split), or per
//     sub-split of 2048 .. 256 samples when that leaves the GPU idle:
//     tcgen05 kind::f16 MMAs over the split's 4 096 samples, both operands
//     staged by TMA through a 3-stage ring, hi.hi' + hi.lo' + lo.hi' into
//     128 x 128 float32 TMEM accumulators, 256 samples each, added up in
//     registers, then written (times 2^-(e_i + e_j), exact) as the split's
//     partial product.  No single sum adds more than 4 096 products, the page's
//     reason for the splits.
//  4. sum: every output entry (a thread each) adds its S partials in float64, in split
//     order, adds back the centring for the second moment (in float64),
//     divides by the true sample count n and writes or adds the float32
//     result; entry (i, j) and (j, i) both read the partial of (min, max),
//     so the result is exactly symmetric.
#include <cuda.h>
#include <cuda_fp16.h>

#include <climits>
#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tc_pipe.cuh"

namespace hdbmst {

namespace {

using namespace tc;

constexpr int kWords = kMomentSplit / 2;         // 32-bit words (two halves) per split row
constexpr int kMomSlabs = kWords / kSlab;         // 64 slabs of 64 halves
constexpr int kMomStages = 3;
constexpr uint32_t kMomStage = 4 * kSlabTile;     // A hi, A lo, B hi, B lo
constexpr size_t kMomSmem = kMomStages * kMomStage + 1024;
constexpr int kMomThreads = 6 * 32;               // producer, MMA, four epilogue warps

constexpr int kStatsThreads = 1024;

__device__ __forceinline__ void kahan_add(float &sum, float &comp, float x) {
    const float y = __fsub_rn(x, comp);
    const float u = __fadd_rn(sum, y);
    comp = __fsub_rn(__fsub_rn(u, sum), y);
    sum = u;
}

__global__ void __launch_bounds__(kStatsThreads) moment_stats_kernel(
    const float *__restrict__ X, int64_t ld, int64_t t0, int64_t n, double *__restrict__ sum,
    float *__restrict__ mu_hi, float *__restrict__ mu_lo, int *__restrict__ scale_e,
    MomentStatus *__restrict__ st) {
    __shared__ double red[kStatsThreads / 32];
    __shared__ unsigned redm[kStatsThreads / 32];
    const int c = blockIdx.x, tid = threadIdx.x;
    const float *row = X + static_cast<int64_t>(c) * ld + t0;
    // two compensated float32 sums per thread (samples t and t + stride,
    // interleaved), then float64 across threads in a fixed order
    float s0 = 0.f, c0 = 0.f, s1 = 0.f, c1 = 0.f, amax = 0.f;
    const int64_t stride = 2 * static_cast<int64_t>(kStatsThreads);
    int64_t t = tid;
    for (; t + kStatsThreads < n; t += stride) {
        const float x0 = row[t], x1 = row[t + kStatsThreads];
        amax = fmaxf(amax, fmaxf(fabsf(x0), fabsf(x1)));
        kahan_add(s0, c0, x0);
        kahan_add(s1, c1, x1);
    }
    if (t < n) {
        const float x0 = row[t];
        amax = fmaxf(amax, fabsf(x0));
        kahan_add(s0, c0, x0);
    }
    double acc = (static_cast<double>(s0) - static_cast<double>(c0)) +
                 (static_cast<double>(s1) - static_cast<double>(c1));
    unsigned m = isfinite(amax) ? __float_as_uint(amax) : 0x7f800000u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        acc += __shfl_xor_sync(0xffffffffu, acc, o);
        m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    }
    if ((tid & 31) == 0) {
        red[tid >> 5] = acc;
        redm[tid >> 5] = m;
    }
    __syncthreads();
    if (tid == 0) {
        double sm = 0.0;
        unsigned mm = 0u;
        for (int w = 0; w < kStatsThreads / 32; ++w) {
            sm += red[w];
            mm = max(mm, redm[w]);
        }
        const double mu = sm / static_cast<double>(n);
        const float h = static_cast<float>(mu);
        sum[c] = sm;
        mu_hi[c] = h;
        mu_lo[c] = static_cast<float>(mu - static_cast<double>(h));
        if (mm >= 0x7f800000u || !isfinite(mu)) atomicOr(&st->status, kStatusNonFinite);
        // the channel's power-of-two scale: its centred values are at most
        // max |x| + |mu| (rounded up)
        const float b = __fadd_ru(__uint_as_float(mm), __fmul_ru(fabsf(h), 1.0000002f));
        scale_e[c] = f16_scale_exp(__float_as_uint(b));
    }
}

// f16_split (common.cuh) of two values at once, packed as the operand words
// hold them (the first value in the low half): hi = fp16(x 2^e),
// lo = fp16(x 2^e - hi), each flushed to zero below 2^-14; the paired
// conversions give the same halves as the single ones.
__device__ __forceinline__ void f16_split2(float x0, float x1, float scale, uint32_t &hw,
                                           uint32_t &lw) {
    const float s0 = __fmul_rn(x0, scale), s1 = __fmul_rn(x1, scale);
    float2 h = __half22float2(__floats2half2_rn(s0, s1));
    h.x = fabsf(h.x) < 0x1p-14f ? 0.f : h.x;
    h.y = fabsf(h.y) < 0x1p-14f ? 0.f : h.y;
    float2 l = __half22float2(__floats2half2_rn(__fsub_rn(s0, h.x), __fsub_rn(s1, h.y)));
    l.x = fabsf(l.x) < 0x1p-14f ? 0.f : l.x;
    l.y = fabsf(l.y) < 0x1p-14f ? 0.f : l.y;
    const __half2 hh = __floats2half2_rn(h.x, h.y), ll = __floats2half2_rn(l.x, l.y);
    hw = *reinterpret_cast<const uint32_t *>(&hh);
    lw = *reinterpret_cast<const uint32_t *>(&ll);
}

// grid: (kWords / 256 word blocks, c_pad channels, split blocks); a
// thread makes one 32-bit word (two halves) of each split it visits
__global__ void __launch_bounds__(256) moment_split_kernel(
    const float *__restrict__ X, int64_t ld, int C, int c_pad, int64_t t0, int64_t n, int S,
    const float *__restrict__ mu_hi, const float *__restrict__ mu_lo,
    const int *__restrict__ scale_e, uint32_t *__restrict__ hi, uint32_t *__restrict__ lo) {
    const int wd = blockIdx.x * blockDim.x + threadIdx.x;  // word within the split row
    const int r = blockIdx.y;
    const bool ch = r < C;
    const float scale = ch ? ldexpf(1.f, scale_e[r]) : 1.f;
    const float mh = ch ? mu_hi[r] : 0.f, ml = ch ? mu_lo[r] : 0.f;
    const float *row = X + static_cast<int64_t>(ch ? r : 0) * ld + t0;
    for (int s = blockIdx.z; s < S; s += gridDim.z) {
        const int64_t t = static_cast<int64_t>(s) * kMomentSplit + 2 * wd;  // sample in the window
        const float v0 = (ch && t < n) ? __fsub_rn(__fsub_rn(row[t], mh), ml) : 0.f;
        const float v1 = (ch && t + 1 < n) ? __fsub_rn(__fsub_rn(row[t + 1], mh), ml) : 0.f;
        uint32_t hw, lw;
        f16_split2(v0, v1, scale, hw, lw);
        const int64_t w = (static_cast<int64_t>(s) * c_pad + r) * kWords + wd;
        hi[w] = hw;
        lo[w] = lw;
    }
}

constexpr int kChunkSlabs = 4;                    // 256 samples per TMEM accumulation
constexpr int kEpiThreads = 4 * 32;
constexpr int kMaxSub = kMomSlabs / kChunkSlabs;  // sub-splits of a split: at most 16

struct MomSmem {
    uint64_t full[kMomStages], empty[kMomStages], afull[2], aempty[2];
    uint32_t tmem_base;
    int abort;
    int last_load[kMomStages];  // slab last loaded into each stage (-1: none)
    int last_mma;               // slab whose MMAs were committed last (-1: none)
};

struct MomParams {
    CUtensorMap hi, lo;  // [S * c_pad rows][kWords words], boxes of 128 rows x 32 words
    float *partial;      // [S * sub][c_pad][c_pad]
    int c_pad, blocks;
    int sub;             // CTAs per split, each over 64 / sub slabs
    const int *scale_e;  // [c_pad] per-channel exponents (0 for padding)
    unsigned *status;
};

// One CTA per (tile pair, split).  The split's 64 slabs go through a
// 3-stage TMA ring; the MMAs of every 4 slabs (256 samples) accumulate in one
// of two TMEM accumulators, alternately, and the epilogue adds each chunk's
// 128 x 128 result into float32 registers while the next chunk is
// multiplied.  Short TMEM accumulations keep the rounding of the running
// accumulator from building up along the split (measured: one accumulation
// over all 4 096 samples left the same-sign sums of a variance 3e-5 low).
__global__ void __launch_bounds__(kMomThreads, 1) moment_product_kernel(
    const __grid_constant__ MomParams P) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ MomSmem S;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // tile pair (I, J), I <= J, numbered row by row
    int p = blockIdx.x, I = 0;
    while (I < P.blocks && p >= P.blocks - I) {
        p -= P.blocks - I;
        ++I;
    }
    const int J = I + p;
    const int s = blockIdx.y / P.sub, part = blockIdx.y % P.sub;
    const int nslabs = kMomSlabs / P.sub, slab0 = part * nslabs, nchunks = nslabs / kChunkSlabs;
    const bool diag = I == J;
    const int rowA = s * P.c_pad + I * kRows, rowB = s * P.c_pad + J * kRows;
    const uint32_t sb = smem_u32(pipe_base(smem_raw));
    if (tid == 0) {
        for (int i = 0; i < kMomStages; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], 1);
            S.last_load[i] = -1;
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&S.afull[i], 1);
            mbar_init(&S.aempty[i], kEpiThreads);
        }
        S.abort = 0;
        S.last_mma = -1;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&S.tmem_base, 256);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = S.tmem_base;
    if (warp == 0 && lane == 0) {
        // producer: the split's 64 slabs of rows I (and J), hi and lo parts
        const uint32_t bytes = (diag ? 2u : 4u) * kSlabTile;
        for (int k = 0; k < nslabs; ++k) {
            const int st = k % kMomStages;
            const uint32_t par = static_cast<uint32_t>(k / kMomStages) & 1u;
            if (!mbar_wait<kSleepProducer>(&S.empty[st], par ^ 1u) ||
                *reinterpret_cast<volatile int *>(&S.abort)) {
                S.abort = 1;
                break;
            }
            const uint32_t a = sb + st * kMomStage;
            const int x = (slab0 + k) * kSlab;
            mbar_expect_tx(&S.full[st], bytes);
            tma_load_2d(a, &P.hi, x, rowA, &S.full[st]);
            tma_load_2d(a + kSlabTile, &P.lo, x, rowA, &S.full[st]);
            if (!diag) {
                tma_load_2d(a + 2 * kSlabTile, &P.hi, x, rowB, &S.full[st]);
                tma_load_2d(a + 3 * kSlabTile, &P.lo, x, rowB, &S.full[st]);
            }
            S.last_load[st] = k;
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer: per slab 4 K steps of 16 halves, three products each
        const uint32_t idesc = instr_desc_f16(kRows, kRows);
        bool ok = true;
        for (int k = 0; k < nslabs && ok; ++k) {
            const int c = k / kChunkSlabs, acc = c & 1;
            const uint32_t d = tmem + static_cast<uint32_t>(acc * kRows);
            if (k % kChunkSlabs == 0 && c >= 2) {
                // the epilogue has taken chunk c - 2 out of this accumulator
                ok = mbar_wait<kSleepMma>(&S.aempty[acc], static_cast<uint32_t>(c / 2 - 1) & 1u);
                if (!ok) break;
                fence_after();
            }
            const int st = k % kMomStages;
            const uint32_t par = static_cast<uint32_t>(k / kMomStages) & 1u;
            ok = mbar_wait<kSleepMma>(&S.full[st], par) &&
                 !*reinterpret_cast<volatile int *>(&S.abort);
            if (!ok) break;
            fence_after();
            const uint32_t a = sb + st * kMomStage;
            const uint64_t ah = smem_desc(a), al = smem_desc(a + kSlabTile);
            const uint64_t bh = diag ? ah : smem_desc(a + 2 * kSlabTile);
            const uint64_t bl = diag ? al : smem_desc(a + 3 * kSlabTile);
#pragma unroll
            for (int kk = 0; kk < kSlab / 8; ++kk) {
                const uint32_t first = (k % kChunkSlabs == 0 && kk == 0) ? 0u : 1u;
                mma_f16_ss(d, ah + 2 * kk, bh + 2 * kk, idesc, first);
                mma_f16_ss(d, ah + 2 * kk, bl + 2 * kk, idesc, 1u);
                mma_f16_ss(d, al + 2 * kk, bh + 2 * kk, idesc, 1u);
            }
            mma_commit(&S.empty[st]);
            S.last_mma = k;
            if (k % kChunkSlabs == kChunkSlabs - 1) mma_commit(&S.afull[acc]);
        }
        if (!ok) S.abort = 1;
    } else if (warp >= 2) {
        // epilogue: warp w reads TMEM lanes 32 (w % 4) .. (its 32 rows of I)
        const int q = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        float sum[kRows];
#pragma unroll
        for (int j = 0; j < kRows; ++j) sum[j] = 0.f;
        bool ok = true;
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
            const int acc = c & 1;
            const bool w = mbar_wait<kSleepEpilogue>(&S.afull[acc], static_cast<uint32_t>(c / 2) & 1u);
            if (!w) S.abort = 1;
            // a warp leaves together: tcgen05.ld is warp-collective
            if (__any_sync(0xffffffffu, !w || *reinterpret_cast<volatile int *>(&S.abort))) {
                ok = false;
                break;
            }
            fence_after();
#pragma unroll
            for (int cc = 0; cc < kRows / 32; ++cc) {
                float v[32];
                tmem_ld32(tmem + lane_base + static_cast<uint32_t>(acc * kRows + cc * 32), v);
#pragma unroll
                for (int j = 0; j < 32; ++j) sum[cc * 32 + j] += v[j];
            }
            fence_before();
            mbar_arrive(&S.aempty[acc]);
        }
        if (ok) {
            // undo the two channels' scales: 2^-(e_row + e_col), exact
            const int row = q * 32 + lane;
            const int er = P.scale_e[I * kRows + row];
            const int *ec = P.scale_e + J * kRows;
            float *dst = P.partial + (static_cast<int64_t>(blockIdx.y) * P.c_pad + I * kRows + row) *
                                         P.c_pad + J * kRows;
#pragma unroll
            for (int j4 = 0; j4 < kRows / 4; ++j4)
                *reinterpret_cast<float4 *>(dst + j4 * 4) = make_float4(
                    ldexpf(sum[j4 * 4], -(er + ec[j4 * 4])), ldexpf(sum[j4 * 4 + 1], -(er + ec[j4 * 4 + 1])),
                    ldexpf(sum[j4 * 4 + 2], -(er + ec[j4 * 4 + 2])),
                    ldexpf(sum[j4 * 4 + 3], -(er + ec[j4 * 4 + 3])));
        }
    }
    // teardown: after a give-up, drain the copies and products still in
    // flight (bounded waits), then free TMEM
    fence_before();
    __syncthreads();
    if (S.abort && tid == 0) {
        atomicOr(P.status, kStatusTimeout);
        for (int i = 0; i < kMomStages; ++i)
            if (S.last_load[i] >= 0)
                mbar_wait<kSleepProducer>(&S.full[i],
                                          static_cast<uint32_t>(S.last_load[i] / kMomStages) & 1u);
        if (S.last_mma >= 0)
            mbar_wait<kSleepProducer>(&S.empty[S.last_mma % kMomStages],
                                      static_cast<uint32_t>(S.last_mma / kMomStages) & 1u);
    }
    __syncthreads();
    fence_after();
    if (warp == 1) tmem_free(tmem, 256);
}

// Sum of the splits: one thread per output entry (i, j) adds the partials of
// (min(i, j), max(i, j)) over the splits in float64, in order (so (i, j) and
// (j, i) get the same bits), and for the second moment adds back what the
// centring took out: with v = x - mu' and s = sum_t v = sum_t x - n mu',
// sum_t x_i x_j = sum_t v_i v_j + mu'_i s_j + mu'_j s_i + n mu'_i mu'_j
// (exact algebra for any offset mu').  Then it divides by n and writes (or
// adds) the float32 result.
__global__ void __launch_bounds__(256) moment_sum_kernel(const float *__restrict__ partial, int S,
                                                         int c_pad, int C, int64_t n, int centred,
                                                         const double *__restrict__ sum,
                                                         const float *__restrict__ mu_hi,
                                                         const float *__restrict__ mu_lo,
                                                         int accumulate, float *__restrict__ out) {
    const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= static_cast<int64_t>(C) * C) return;
    const int i = static_cast<int>(e / C), j = static_cast<int>(e % C);
    const int a = min(i, j), b = max(i, j);
    const float *p = partial + static_cast<int64_t>(a) * c_pad + b;
    const int64_t plane = static_cast<int64_t>(c_pad) * c_pad;
    double acc = 0.0;
    int s = 0;
    for (; s + 4 <= S; s += 4) {
        const float p0 = p[s * plane], p1 = p[(s + 1) * plane], p2 = p[(s + 2) * plane],
                    p3 = p[(s + 3) * plane];
        acc += static_cast<double>(p0);
        acc += static_cast<double>(p1);
        acc += static_cast<double>(p2);
        acc += static_cast<double>(p3);
    }
    for (; s < S; ++s) acc += static_cast<double>(p[s * plane]);
    const double dn = static_cast<double>(n);
    if (!centred) {
        const double mi = static_cast<double>(mu_hi[i]) + static_cast<double>(mu_lo[i]);
        const double mj = static_cast<double>(mu_hi[j]) + static_cast<double>(mu_lo[j]);
        const double si = sum[i] - dn * mi, sj = sum[j] - dn * mj;
        // the same float64 operations for (i, j) and (j, i): symmetric
        acc += min(mi * sj, mj * si) + max(mi * sj, mj * si) + dn * (mi * mj);
    }
    const float f = static_cast<float>(acc / dn);
    out[e] = accumulate ? out[e] + f : f;
}

}  // namespace

bool moment_supported() { return tensor_maps_available(); }

int moment_splits(int64_t n) { return static_cast<int>((n + kMomentSplit - 1) / kMomentSplit); }

cudaError_t launch_moment_stats(const float *X, int64_t ld, int C, int64_t t0, int64_t n,
                                double *sum, float *mu_hi, float *mu_lo, int *scale_e,
                                MomentStatus *st, cudaStream_t s) {
    moment_stats_kernel<<<C, kStatsThreads, 0, s>>>(X, ld, t0, n, sum, mu_hi, mu_lo, scale_e, st);
    return cudaGetLastError();
}

cudaError_t launch_moment_split(const float *X, int64_t ld, int C, int c_pad, int64_t t0,
                                int64_t n, const float *mu_hi, const float *mu_lo,
                                const int *scale_e, uint32_t *hi, uint32_t *lo, cudaStream_t s) {
    const int S = moment_splits(n);
    const dim3 grid(kWords / 256, c_pad, std::min(S, 65535));
    moment_split_kernel<<<grid, 256, 0, s>>>(X, ld, C, c_pad, t0, n, S, mu_hi, mu_lo, scale_e, hi,
                                             lo);
    return cudaGetLastError();
}

int moment_subsplits(int c_pad, int64_t n) {
    const int64_t pairs = static_cast<int64_t>(c_pad / kRows) * (c_pad / kRows + 1) / 2;
    const int64_t ctas = pairs * moment_splits(n);
    int sub = 1;
    while (sub < kMaxSub && ctas * sub * 2 <= kMomentTargetCtas) sub *= 2;
    return sub;
}

cudaError_t launch_moment_product(const uint32_t *hi, const uint32_t *lo, int c_pad, int64_t n,
                                  const int *scale_e, float *partial, unsigned *status,
                                  cudaStream_t s) {
    const int S = moment_splits(n);
    MomParams P{};
    const int64_t rows = static_cast<int64_t>(S) * c_pad;
    if (!make_point_map(&P.hi, reinterpret_cast<const float *>(hi), rows, kWords) ||
        !make_point_map(&P.lo, reinterpret_cast<const float *>(lo), rows, kWords))
        return cudaErrorInvalidValue;
    P.partial = partial;
    P.c_pad = c_pad;
    P.blocks = c_pad / kRows;
    P.sub = moment_subsplits(c_pad, n);
    P.scale_e = scale_e;
    P.status = status;
    cudaError_t e = cudaFuncSetAttribute(moment_product_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kMomSmem));
    if (e != cudaSuccess) return e;
    const int pairs = P.blocks * (P.blocks + 1) / 2;
    moment_product_kernel<<<dim3(pairs, S * P.sub), kMomThreads, kMomSmem, s>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_moment_sum(const float *partial, int c_pad, int C, int64_t n, int centred,
                              const double *sum, const float *mu_hi, const float *mu_lo,
                              int accumulate, float *out, cudaStream_t s) {
    const int64_t entries = static_cast<int64_t>(C) * C;
    moment_sum_kernel<<<static_cast<int>((entries + 255) / 256), 256, 0, s>>>(
        partial, moment_splits(n) * moment_subsplits(c_pad, n), c_pad, C, n, centred, sum, mu_hi,
        mu_lo, accumulate, out);
    return cudaGetLastError();
}

cudaError_t moment_test_hooks(unsigned long long wait_ns, int withhold) {
    return tc::set_test_hooks(wait_ns, withhold);
}

}  // namespace hdbmst
