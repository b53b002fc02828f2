// kvq8_device.cuh -- device-side helpers shared by the kvq8 kernels: warp
// reductions and the two quantisation rules, written once so that the
// stand-alone query quantiser and the decode prologue run the same code.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq8.h"

namespace kvq8 {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void flag_status(uint32_t *status, uint32_t bits) {
    if (status) atomicOr(status, bits);
}

// 1/127 rounded to fp32 (the pages' KVQ_INV); folded at compile time with
// IEEE round-to-nearest.
#define KVQ8_INV127 (1.0f / 127.0f)

// Per-(token, head) K/V rule ([Day 9-3] §2): given the row's max |v| (already
// reduced), scale = max/127 and code = round_half_even(v/scale) in [-127, 127].
// The intrinsics pin IEEE division and rounding; nothing here may be fused.
__device__ __forceinline__ float kv_row_scale(float max_abs) {
    return __fdiv_rn(max_abs, 127.0f);
}

__device__ __forceinline__ int kv_code(float v, float scale) {
    if (scale == 0.0f) return 0;
    int c = __float2int_rn(__fdiv_rn(v, scale));
    return max(-127, min(127, c));
}

// kv_code of four values of one row whose scale is sc = fl(max|row| / 127),
// each in the low byte of a word, with one reciprocal per row in place of a
// division per value.  inv approximates 1 / sc (the hardware reciprocal, which
// the PTX ISA bounds by one ulp; the argument below allows three).  t =
// fl(v * inv + 1.5 * 2^23) holds round_half_even(v * inv) in its low mantissa
// bits (the sum lies where the fp32 spacing is 1, and 1.5 * 2^23 is even), so
// its low byte is the code as a two's complement byte; e = fl(v * inv - r),
// r = t - 1.5 * 2^23, is the residual of that rounding to within 2^-26.  For
// |v| <= max|row|, |v / sc| < 127.0001, so v * inv lies within
// 127.0001 * 3 * 2^-23 < 4.6e-5 of v / sc, and fl(v / sc) within half an ulp
// below 128 (2^-18) of v / sc.  When |e| <= 1/2 - 2^-14 (2^-14 > 6.1e-5 >
// 4.6e-5 + 2^-18 + 2^-26), fl(v / sc) is therefore strictly closer than 1/2
// to r, and round_half_even(fl(v / sc)) = r, which is within [-127, 127] (no
// clamp needed).  The four values are divided exactly when one residual is
// larger (about 1.2e-4 of values) or not a number, or when sc lies outside
// [2^-120, 2^120] (a zero row, a subnormal or non-finite scale); the result
// equals kv_code's in every case.
__device__ __forceinline__ uint4 kv_code_bytes4(float4 x, float sc) {
    if (sc >= 0x1p-120f && sc <= 0x1p120f) {
        constexpr float kShift = 0x1.8p23f;
        constexpr float kLim = 0.5f - 0x1p-14f;
        float inv;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(sc));
        const float t0 = __fmaf_rn(x.x, inv, kShift), t1 = __fmaf_rn(x.y, inv, kShift);
        const float t2 = __fmaf_rn(x.z, inv, kShift), t3 = __fmaf_rn(x.w, inv, kShift);
        const float e0 = __fmaf_rn(x.x, inv, -__fsub_rn(t0, kShift));
        const float e1 = __fmaf_rn(x.y, inv, -__fsub_rn(t1, kShift));
        const float e2 = __fmaf_rn(x.z, inv, -__fsub_rn(t2, kShift));
        const float e3 = __fmaf_rn(x.w, inv, -__fsub_rn(t3, kShift));
        if ((fabsf(e0) <= kLim) & (fabsf(e1) <= kLim) & (fabsf(e2) <= kLim) & (fabsf(e3) <= kLim))
            return make_uint4(__float_as_uint(t0), __float_as_uint(t1), __float_as_uint(t2),
                              __float_as_uint(t3));
    }
    return make_uint4((uint32_t)kv_code(x.x, sc), (uint32_t)kv_code(x.y, sc),
                      (uint32_t)kv_code(x.z, sc), (uint32_t)kv_code(x.w, sc));
}

// The low bytes of four words as one little-endian word.
__device__ __forceinline__ uint32_t low_bytes4(uint4 c) {
    return __byte_perm(__byte_perm(c.x, c.y, 0x0040), __byte_perm(c.z, c.w, 0x0040), 0x5410);
}

// True when v is a NaN or an infinity (all exponent bits set).
__device__ __forceinline__ bool nonfinite(float v) {
    return (__float_as_uint(v) & 0x7f800000u) == 0x7f800000u;
}

// Scale of a K/V row held as a float4 per lane (lane l: dims 4l..4l+3) by the
// rule above, with the reading taken for values the pages do not cover: a row
// holding a NaN or an infinity is quantised as a row of zeros (x is cleared,
// scale 0, so every code is 0) and KVQ8_DEV_NONFINITE is set.  |v| as a bit
// pattern: non-negative floats order like their bit patterns, infinity above
// every finite value and NaN above infinity, so one unsigned warp reduction
// gives both the row maximum and the test.
__device__ __forceinline__ float kv_row_scale_checked(float4 &x, uint32_t *status) {
    const uint32_t a = max(max(__float_as_uint(x.x) & 0x7fffffffu, __float_as_uint(x.y) & 0x7fffffffu),
                           max(__float_as_uint(x.z) & 0x7fffffffu, __float_as_uint(x.w) & 0x7fffffffu));
    const uint32_t m = __reduce_max_sync(0xffffffffu, a);
    if (m >= 0x7f800000u) {   // warp-uniform
        x = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if ((threadIdx.x & 31) == 0) flag_status(status, KVQ8_DEV_NONFINITE);
        return 0.0f;
    }
    return kv_row_scale(__uint_as_float(m));
}

// 32-block query rule ([Day 9-2] §2 segment 1) for one row of 128 values,
// executed by one full warp: lane l holds element 32*k + l of block k in x[k].
// qm = max |x| over the block (1 when below 1e-6); block scale = qm * (1/127);
// code = round_half_even(x * (127/qm)) clamped to [-128, 127].  A block that
// holds a NaN or an infinity is quantised as a block of zeros (scale 1/127,
// codes 0) and KVQ8_DEV_NONFINITE is set in *status (when non-null).  The
// four block maxima are four independent unsigned warp reductions of |x| as
// bit patterns (the order of kv_row_scale_checked), which also detect the
// non-finite blocks.
__device__ __forceinline__ void quantize_q_vals_warp(const float (&xs)[4], int lane, int8_t *codes,
                                                     float *scales, uint32_t *status) {
    uint32_t mb[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) mb[k] = __reduce_max_sync(0xffffffffu, __float_as_uint(xs[k]) & 0x7fffffffu);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float x = xs[k];
        float qm;
        if (mb[k] >= 0x7f800000u) {   // warp-uniform
            x = 0.0f;
            qm = 1.0f;
            if (lane == 0) flag_status(status, KVQ8_DEV_NONFINITE);
        } else {
            qm = __uint_as_float(mb[k]);
            if (qm < 1e-6f) qm = 1.0f;
        }
        const float iq = __fdiv_rn(127.0f, qm);
        int c = __float2int_rn(__fmul_rn(x, iq));
        c = max(-128, min(127, c));
        codes[32 * k + lane] = (int8_t)c;
        if (lane == 0) scales[k] = __fmul_rn(qm, KVQ8_INV127);
    }
}

// The same for a row in global memory.
__device__ __forceinline__ void quantize_q_row_warp(const float *__restrict__ row, int lane,
                                                    int8_t *codes, float *scales, uint32_t *status) {
    float xs[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) xs[k] = row[32 * k + lane];
    quantize_q_vals_warp(xs, lane, codes, scales, status);
}

}  // namespace kvq8
