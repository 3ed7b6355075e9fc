// K0: pack a caller point set into the library's padded layouts and compute
// squared norms.
//
// The caller's set is feature-major [d, n] with any leading dimension; the
// distance tiles want rows padded to the tile width with 16-byte-aligned
// strides, and the exact re-evaluation wants each point's features
// contiguous.  One pass writes both copies and the norm |x|^2 that the
// expansion |x|^2 + |y|^2 - 2 x.y needs (page "Kilosort4 clustering and
// matching", gpu/clustering, "k-nearest neighbours are a matrix product").
// Padding features and padding points are zero; a padding point's norm is
// +inf so that it never ranks as a neighbour.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace hdbmst {

namespace {

__global__ void __launch_bounds__(256) pack_kernel(const float *__restrict__ X, int64_t ld, int n,
                                                   int d, int n_pad, int dk,
                                                   float *__restrict__ Xf,
                                                   float *__restrict__ Xp,
                                                   float *__restrict__ Xlo,
                                                   float *__restrict__ norm,
                                                   unsigned *__restrict__ status,
                                                   unsigned *__restrict__ nbmax_bits,
                                                   const int *__restrict__ perm,
                                                   uint2 *__restrict__ Xh16,
                                                   uint2 *__restrict__ Xl16,
                                                   const unsigned *__restrict__ amax_bits,
                                                   float *__restrict__ e0_out,
                                                   const int *__restrict__ inv,
                                                   float *__restrict__ Xhi) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const bool inside = i < n_pad;
    const bool valid = i < n;
    // perm: thread i writes position i from the caller's point perm[i]; inv:
    // thread i reads the caller's point i (coalesced) and writes position
    // inv[i] (rows of dk floats are contiguous; Xf is then not written)
    const int src = (valid && perm) ? perm[i] : i;
    const int dst = (valid && inv) ? inv[i] : i;
    float acc = 0.f;
    bool finite = true;
    // two-part FP16 operands: the set's scale 2^e (an exact power of two)
    const float scale = Xh16 ? ldexpf(1.f, f16_scale_exp(*amax_bits)) : 1.f;
    // the FP16 form's absolute error part, once per call for every proof
    if (Xh16 && e0_out && i == 0) *e0_out = __double2float_ru(f16_abs_err(true, dk, *amax_bits));
    if (inside) {
        for (int f = 0; f < dk; f += 4) {
            float v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int ff = f + q;
                v[q] = (valid && ff < d) ? X[static_cast<int64_t>(ff) * ld + src] : 0.f;
                finite = finite && isfinite(v[q]);
                if (Xf) Xf[static_cast<int64_t>(ff) * n_pad + dst] = v[q];
                acc = __fmaf_rn(v[q], v[q], acc);
            }
            if (Xp)
                *reinterpret_cast<float4 *>(Xp + static_cast<int64_t>(dst) * dk + f) =
                    make_float4(v[0], v[1], v[2], v[3]);
            if (Xlo) {
                // the tensor-core tile's two operand parts: hi = x cut to its top
                // 19 bits (a TF32 value, exact whatever rounding the MMA applies
                // to its inputs) and lo = x - hi (exact in float32)
                float hh[4], l[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    hh[q] = tf32_trunc(v[q]);
                    l[q] = __fsub_rn(v[q], hh[q]);
                }
                const int64_t e = static_cast<int64_t>(dst) * dk + f;
                *reinterpret_cast<float4 *>(Xhi + e) = make_float4(hh[0], hh[1], hh[2], hh[3]);
                *reinterpret_cast<float4 *>(Xlo + e) = make_float4(l[0], l[1], l[2], l[3]);
            }
            if (Xh16) {
                // four halves = two 32-bit words, lower feature in the low half
                unsigned short h[4], l[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) f16_split(v[q], scale, h[q], l[q]);
                const int64_t o = (static_cast<int64_t>(dst) * dk + f) / 4;
                Xh16[o] = make_uint2(h[0] | (static_cast<unsigned>(h[1]) << 16),
                                     h[2] | (static_cast<unsigned>(h[3]) << 16));
                Xl16[o] = make_uint2(l[0] | (static_cast<unsigned>(l[1]) << 16),
                                     l[2] | (static_cast<unsigned>(l[3]) << 16));
            }
        }
        norm[dst] = valid ? acc : INFINITY;
    }
    if (!finite) atomicOr(status, kStatusNonFinite);
    // largest norm over valid points: warp maximum, one atomic per warp
    unsigned bits = valid ? __float_as_uint(acc) : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bits = max(bits, __shfl_xor_sync(0xffffffffu, bits, o));
    if ((threadIdx.x & 31) == 0 && nbmax_bits && bits) atomicMax(nbmax_bits, bits);
}

// The same outputs as pack_kernel (without perm), staged through shared
// memory: a CTA takes 32 points, reads 64 features at a time with coalesced
// rows of the caller's feature-major set, then half-warps write each point's
// point-major rows (256 bytes of floats, 128 bytes of halves) contiguously.
// Each point's norm is the same ascending-feature chain of fused
// multiply-adds as in pack_kernel, so the bits agree.
constexpr int kPackPts = 32, kPackF = 64;
__global__ void __launch_bounds__(256) pack_tile_kernel(const float *__restrict__ X, int64_t ld,
                                                        int n, int d, int n_pad, int dk,
                                                        float *__restrict__ Xf,
                                                        float *__restrict__ Xp,
                                                        float *__restrict__ Xlo,
                                                        float *__restrict__ norm,
                                                        unsigned *__restrict__ status,
                                                        unsigned *__restrict__ nbmax_bits,
                                                        uint2 *__restrict__ Xh16,
                                                        uint2 *__restrict__ Xl16,
                                                        const unsigned *__restrict__ amax_bits,
                                                        float *__restrict__ e0_out,
                                                        const int *__restrict__ inv,
                                                        float *__restrict__ Xhi) {
    __shared__ float xs[kPackF][kPackPts + 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int i0 = blockIdx.x * kPackPts;
    const float scale = Xh16 ? ldexpf(1.f, f16_scale_exp(*amax_bits)) : 1.f;
    if (Xh16 && e0_out && blockIdx.x == 0 && tid == 0)
        *e0_out = __double2float_ru(f16_abs_err(true, dk, *amax_bits));
    float acc = 0.f;  // warp 0: point i0 + lane
    bool finite = true;
    const int ip = i0 + lane;
    const int dst_own = (ip < n && inv) ? inv[ip] : ip;
    // warp w stages features w, w + 8, ... of the chunk: all eight loads in
    // flight at once, the next chunk's while this one is written
    constexpr int kRows = kPackF / 8;
    float vr[kRows];
    const auto load_chunk = [&](int f0) {
#pragma unroll
        for (int u = 0; u < kRows; ++u) {
            const int f = f0 + warp + 8 * u;
            vr[u] = (f < d && f < dk && ip < n) ? X[static_cast<int64_t>(f) * ld + ip] : 0.f;
        }
    };
    load_chunk(0);
    for (int f0 = 0; f0 < dk; f0 += kPackF) {
        const int fc = min(kPackF, dk - f0);
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kRows; ++u) {
            const int r = warp + 8 * u;
            if (r < fc) {
                xs[r][lane] = vr[u];
                if (Xf && ip < n_pad) Xf[static_cast<int64_t>(f0 + r) * n_pad + dst_own] = vr[u];
            }
        }
        __syncthreads();
        if (f0 + kPackF < dk) load_chunk(f0 + kPackF);
        if (warp == 0) {
            for (int r = 0; r < fc; ++r) {
                const float v = xs[r][lane];
                finite = finite && isfinite(v);
                acc = __fmaf_rn(v, v, acc);
            }
        }
        // half-warp h of warp w: points 2 w + h, + 16, ...; lane c: features 4c .. 4c + 3
        const int c = lane & 15;
        for (int q = warp * 2 + (lane >> 4); q < kPackPts; q += 16) {
            const int i = i0 + q;
            if (4 * c >= fc || i >= n_pad) continue;
            const int dst = (i < n && inv) ? inv[i] : i;
            const float v0 = xs[4 * c][q], v1 = xs[4 * c + 1][q], v2 = xs[4 * c + 2][q],
                        v3 = xs[4 * c + 3][q];
            const int64_t e = static_cast<int64_t>(dst) * dk + f0 + 4 * c;
            if (Xp) *reinterpret_cast<float4 *>(Xp + e) = make_float4(v0, v1, v2, v3);
            if (Xlo) {
                const float h0 = tf32_trunc(v0), h1 = tf32_trunc(v1), h2 = tf32_trunc(v2),
                            h3 = tf32_trunc(v3);
                *reinterpret_cast<float4 *>(Xhi + e) = make_float4(h0, h1, h2, h3);
                *reinterpret_cast<float4 *>(Xlo + e) =
                    make_float4(__fsub_rn(v0, h0), __fsub_rn(v1, h1), __fsub_rn(v2, h2),
                                __fsub_rn(v3, h3));
            }
            if (Xh16) {
                unsigned short h0, h1, h2, h3, lo0, lo1, lo2, lo3;
                f16_split(v0, scale, h0, lo0);
                f16_split(v1, scale, h1, lo1);
                f16_split(v2, scale, h2, lo2);
                f16_split(v3, scale, h3, lo3);
                Xh16[e / 4] = make_uint2(h0 | (static_cast<unsigned>(h1) << 16),
                                         h2 | (static_cast<unsigned>(h3) << 16));
                Xl16[e / 4] = make_uint2(lo0 | (static_cast<unsigned>(lo1) << 16),
                                         lo2 | (static_cast<unsigned>(lo3) << 16));
            }
        }
    }
    if (warp == 0) {
        const bool valid = ip < n;
        if (ip < n_pad) norm[dst_own] = valid ? acc : INFINITY;
        if (!finite) atomicOr(status, kStatusNonFinite);
        unsigned bits = valid ? __float_as_uint(acc) : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bits = max(bits, __shfl_xor_sync(0xffffffffu, bits, o));
        if (lane == 0 && nbmax_bits && bits) atomicMax(nbmax_bits, bits);
    }
}

// Largest magnitude of the caller's [d, n] set, raised into *amax_bits
// (non-negative floats order like their bits; non-finite values are the pack
// kernel's to report).
__global__ void __launch_bounds__(256) absmax_kernel(const float *__restrict__ X, int64_t ld,
                                                     int n, int d,
                                                     unsigned *__restrict__ amax_bits) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    unsigned bits = 0u;
    if (i < n)
        for (int f = 0; f < d; ++f) {
            const float v = fabsf(X[static_cast<int64_t>(f) * ld + i]);
            if (v <= 3.4028234663852886e38f) bits = max(bits, __float_as_uint(v));
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bits = max(bits, __shfl_xor_sync(0xffffffffu, bits, o));
    if ((threadIdx.x & 31) == 0 && bits) atomicMax(amax_bits, bits);
}

__global__ void check_core_kernel(const float *__restrict__ core, int n,
                                  unsigned *__restrict__ status) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        const float c = core[i];
        if (!(isfinite(c) && c >= 0.f)) atomicOr(status, kStatusNonFinite);
    }
}

}  // namespace

cudaError_t launch_pack(const float *X, int64_t ld, int n, int d, int n_pad, int dk, float *Xf,
                        float *Xp, float *Xlo, float *norm, unsigned *status,
                        unsigned *nbmax_bits, cudaStream_t s, const int *perm, uint32_t *Xh16,
                        uint32_t *Xl16, const unsigned *amax_bits, float *e0_out,
                        const int *inv, float *Xhi) {
    if ((Xlo == nullptr) != (Xhi == nullptr)) return cudaErrorInvalidValue;
    if (!perm && dk % 32 == 0) {
        pack_tile_kernel<<<(n_pad + kPackPts - 1) / kPackPts, 256, 0, s>>>(
            X, ld, n, d, n_pad, dk, Xf, Xp, Xlo, norm, status, nbmax_bits,
            reinterpret_cast<uint2 *>(Xh16), reinterpret_cast<uint2 *>(Xl16), amax_bits, e0_out,
            inv, Xhi);
        return cudaGetLastError();
    }
    const int blocks = static_cast<int>((n_pad + 255) / 256);
    pack_kernel<<<blocks, 256, 0, s>>>(X, ld, n, d, n_pad, dk, Xf, Xp, Xlo, norm, status,
                                       nbmax_bits, perm, reinterpret_cast<uint2 *>(Xh16),
                                       reinterpret_cast<uint2 *>(Xl16), amax_bits, e0_out, inv,
                                       Xhi);
    return cudaGetLastError();
}

cudaError_t launch_absmax(const float *X, int64_t ld, int n, int d, unsigned *amax_bits,
                          cudaStream_t s) {
    absmax_kernel<<<(n + 255) / 256, 256, 0, s>>>(X, ld, n, d, amax_bits);
    return cudaGetLastError();
}

cudaError_t launch_check_core(const float *core, int n, unsigned *status, cudaStream_t s) {
    check_core_kernel<<<(n + 255) / 256, 256, 0, s>>>(core, n, status);
    return cudaGetLastError();
}

// The least squared norm of every 32 consecutive points (the tensor-core
// tiles' batches of columns), from norms padded to a multiple of 32 (+inf
// past the last point): one warp per batch.
__global__ void norm_min32_kernel(const float *__restrict__ norm, int64_t n_pad,
                                  float *__restrict__ nmin) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n_pad) return;  // whole warps: n_pad is a multiple of 32
    // non-negative floats (and +inf) order like their bits
    const unsigned m = __reduce_min_sync(0xffffffffu, __float_as_uint(norm[i]));
    if ((threadIdx.x & 31) == 0) nmin[i >> 5] = __uint_as_float(m);
}

cudaError_t launch_norm_min32(const float *norm, int64_t n_pad, float *nmin, cudaStream_t s) {
    if (n_pad <= 0) return cudaSuccess;
    if (n_pad % 32 != 0) return cudaErrorInvalidValue;
    norm_min32_kernel<<<static_cast<unsigned>((n_pad + 255) / 256), 256, 0, s>>>(norm, n_pad, nmin);
    return cudaGetLastError();
}

}  // namespace hdbmst
