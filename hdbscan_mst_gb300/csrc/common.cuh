// Device helpers shared by the kernels of the hdbmst library.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cmath>
#include <cstddef>
#include <cstdint>

namespace hdbmst {

// Distance-tile geometry: a CTA of 256 threads owns 128 rows x 128 columns,
// each thread an 8 x 8 register block; features stream in chunks of 16.
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kBK = 16;
constexpr int kThreads = 256;

// Bits of the device status word.
constexpr unsigned kStatusNonFinite = 1u;
constexpr unsigned kStatusNoConverge = 2u;
constexpr unsigned kStatusOverflow = 4u;
constexpr unsigned kStatusBadList = 8u;
constexpr unsigned kStatusTimeout = 16u;  // a bounded wait on the tensor core gave up

constexpr unsigned long long kNoKey = ~0ull;

__host__ __device__ inline int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

// One feature of the distance every kernel uses: the float32 difference,
// squared and added to the running float32 sum by one fused multiply-add.
// Summed in ascending feature order this is the library's single definition
// of the squared distance (symmetric: a - b and b - a differ only in sign).
__device__ __forceinline__ float sqdiff_fma(float a, float b, float acc) {
    const float t = __fsub_rn(a, b);
    return __fmaf_rn(t, t, acc);
}

// A non-negative float and a 32-bit index packed so that unsigned 64-bit
// order is (value, index) order: non-negative IEEE floats order like their bits.
__device__ __forceinline__ unsigned long long key64(float w, unsigned idx) {
    return (static_cast<unsigned long long>(__float_as_uint(w)) << 32) | idx;
}
__device__ __forceinline__ float key_w(unsigned long long k) {
    return __uint_as_float(static_cast<unsigned>(k >> 32));
}
__device__ __forceinline__ unsigned key_i(unsigned long long k) { return static_cast<unsigned>(k); }

// Order-preserving map of any float (negative ones included) to unsigned.
__device__ __forceinline__ unsigned float_order(float v) {
    const unsigned b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float order_float(unsigned o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// Two-part FP16 operands of the tensor-core tiles (tc.cuh, err_coef_f16).
// The scale 2^e of a point set puts its largest magnitude amax in
// [2^14, 2^15), clamped to |e| <= 60; amax_bits are amax's float bits.
__host__ __device__ inline int f16_scale_exp(unsigned amax_bits) {
    const int E = static_cast<int>((amax_bits >> 23) & 0xffu) - 127;
    const int e = 14 - E;
    return e < -60 ? -60 : (e > 60 ? 60 : e);
}
// Absolute part of the FP16 form's ranking error in t (squared-distance
// units): (2^30 sqrt(dk) + 2 dk) h^2 with h = 2^(-14 - e), 5% slack; zero for
// the other engines.
__host__ __device__ inline double f16_abs_err(bool f16, int dk, unsigned amax_bits) {
    if (!f16) return 0.0;
    const double h = ldexp(1.0, -14 - f16_scale_exp(amax_bits));
    return (0x1p30 * sqrt(static_cast<double>(dk)) + 2.0 * dk) * h * h * 1.05;
}

// x cut to its top 19 bits (sign, exponent, 10 mantissa bits): a TF32 value,
// which a TF32 MMA reads exactly whether it truncates or rounds its inputs;
// x - tf32_trunc(x) is exact in float32 and below 2^-10 |x|.
__device__ __forceinline__ float tf32_trunc(float x) {
    return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// hi, lo halves of x 2^e (scale = 2^e): hi = fp16(x 2^e),
// lo = fp16(x 2^e - hi), each flushed to zero below 2^-14.  x 2^e - hi is
// exact in float32 (hi is x 2^e rounded to fewer bits at no smaller exponent).
__device__ __forceinline__ void f16_split(float x, float scale, unsigned short &hi,
                                          unsigned short &lo) {
    const float xs = __fmul_rn(x, scale);
    float h = __half2float(__float2half_rn(xs));
    if (fabsf(h) < 0x1p-14f) h = 0.f;
    float l = __half2float(__float2half_rn(__fsub_rn(xs, h)));
    if (fabsf(l) < 0x1p-14f) l = 0.f;
    hi = __half_as_ushort(__float2half_rn(h));
    lo = __half_as_ushort(__float2half_rn(l));
}

// The rounding proofs of the refines (knn.cu, scan.cu), in float32 with every
// operation rounded in the safe direction (float64 is slow on this part).
// T = w^2 (1 + 16 u) / (1 - (d + 3) u), u = 2^-24, rounded up; both factors
// are exact floats.
__device__ __forceinline__ float proof_T_up(float w, int d) {
    const float m1 = 1.f + 0x1p-20f;
    const float m2 = 1.f - static_cast<float>(d + 3) * 0x1p-24f;
    return __fdiv_ru(__fmul_ru(__fmul_ru(w, w), m1), m2);
}
// |a|^2 + tau - c (|a|^2 + nb_c) - e0, nb_c = (|a| + sqrt(T))^2, rounded down.
__device__ __forceinline__ float proof_lhs_down(float tau, float na, float T, float c, float e0) {
    const float sq = __fadd_ru(__fsqrt_ru(na), __fsqrt_ru(T));
    const float nbc = __fmul_ru(sq, sq);
    return __fsub_rd(__fsub_rd(__fadd_rd(tau, na), __fmul_ru(c, __fadd_ru(na, nbc))), e0);
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// 16-byte asynchronous global -> shared copy (L2 only), and its group fences.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
// 16 bytes through L1 as well (rows that several warps of the SM read)
__device__ __forceinline__ void cp_async16_ca(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
// 8 bytes (cp.async.cg copies only 16; .ca takes 4, 8 or 16)
__device__ __forceinline__ void cp_async8(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_one() {
    asm volatile("cp.async.wait_group 1;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

}  // namespace hdbmst
