// kvq8_device.cuh -- device-side helpers shared by the kvq8 kernels: warp
// reductions and the two quantisation rules, written once so that the
// stand-alone query quantiser and the decode prologue run the same code.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

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

// 32-block query rule ([Day 9-2] §2 segment 1) for one row of 128 values,
// executed by one full warp: lane l holds element 32*k + l of block k in x[k].
// qm = max |x| over the block (1 when below 1e-6); block scale = qm * (1/127);
// code = round_half_even(x * (127/qm)) clamped to [-128, 127].
__device__ __forceinline__ void quantize_q_vals_warp(const float (&xs)[4], int lane, int8_t *codes,
                                                     float *scales) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float x = xs[k];
        float qm = warp_max(fabsf(x));
        if (qm < 1e-6f) qm = 1.0f;
        const float iq = __fdiv_rn(127.0f, qm);
        int c = __float2int_rn(__fmul_rn(x, iq));
        c = max(-128, min(127, c));
        codes[32 * k + lane] = (int8_t)c;
        if (lane == 0) scales[k] = __fmul_rn(qm, KVQ8_INV127);
    }
}

// The same for a row in global memory.
__device__ __forceinline__ void quantize_q_row_warp(const float *__restrict__ row, int lane,
                                                    int8_t *codes, float *scales) {
    float xs[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) xs[k] = row[32 * k + lane];
    quantize_q_vals_warp(xs, lane, codes, scales);
}

}  // namespace kvq8
