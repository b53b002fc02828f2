// append.cu -- quantise-append of new K/V rows into the paged INT8 cache, and
// the stand-alone 32-block query quantiser.
//
// Quantisation rule: [Day 9-3] §2 and [Day 9-1] §2 (kv_quantize_per_head):
// one fp32 scale = max|v|/127 per (token, kv head) row of 128 values, codes
// round_half_even(v/scale) in [-127, 127].
//
// One CTA takes 32 consecutive new tokens of one (sequence, kv head); each of
// its 8 warps quantises 4 tokens, one row per warp-iteration with a float4 per
// lane (a row is one coalesced 512-byte read).  K codes go straight to the
// token-major K tile (one 128-byte row, its 16-byte chunks permuted by slot);
// V codes are transposed through shared memory so that the dim-major V
// quarters are written as runs of consecutive slots.
#include <limits.h>

#include "kvq8_device.cuh"
#include "kvq8_internal.cuh"
#include "kvq8_ptx.cuh"

namespace kvq8 {
namespace {

constexpr int kAppendTokens = 32;  // tokens per CTA
constexpr int kAppendWarps = 8;
constexpr int kVStride = kAppendTokens + 4;  // bytes per staged V dim row
constexpr int kNoAppend = INT_MIN;            // this sequence appends nothing

// Position of the first new token of sequence b: start_pos[b], or in a decode
// step ctx_lens[b] - 1 (nothing for an empty or out-of-table context, which
// the decode flags).
__device__ __forceinline__ int start_position(const AppendParams &p, int b, int cap) {
    if (p.start_pos) return p.start_pos[b];
    const int L = p.ctx_lens[b];
    return (L >= 1 && L <= cap) ? L - 1 : kNoAppend;
}

__global__ void __launch_bounds__(kAppendWarps * 32)
quantize_append_kernel(AppendParams p) {
    const int h = blockIdx.y, b = blockIdx.z;
    const int i0 = blockIdx.x * kAppendTokens;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    __shared__ __align__(16) int8_t v_stage[kHD][kVStride];
    __shared__ int tok_phys[kAppendTokens];
    __shared__ int tok_slot[kAppendTokens];

    pdl_launch_dependents();  // let the next kernel of the step be scheduled now
    const int cap = p.max_blocks * kBS;
    const int start = start_position(p, b, cap);
    for (int r = warp; r < kAppendTokens; r += kAppendWarps) {
        const int i = i0 + r;
        int phys = -1, slot = 0;
        if (i < p.n_new && start != kNoAppend) {
            const int pos = start + i;
            if (pos < 0 || pos >= cap) {
                if (lane == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_POSITION);
            } else {
                phys = p.block_table[(size_t)b * p.max_blocks + pos / kBS];
                slot = pos % kBS;
                if (phys < 0 || phys >= p.num_blocks) {
                    if (lane == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_BLOCK_ID);
                    phys = -1;
                }
            }
        }
        if (lane == 0) {
            tok_phys[r] = phys;
            tok_slot[r] = slot;
        }
        if (phys < 0) continue;  // warp-uniform

        const size_t src = (((size_t)b * p.n_new + i) * p.nkv + h) * kHD;
        const size_t tile = (size_t)phys * p.nkv + h;

        // K row -> token-major K tile
        {
            const float4 x = reinterpret_cast<const float4 *>(p.k_new + src)[lane];
            float m = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
            m = warp_max(m);
            const float s = kv_row_scale(m);
            const uint32_t w = pack4(kv_code(x.x, s), kv_code(x.y, s), kv_code(x.z, s),
                                     kv_code(x.w, s));
            // 16-byte chunk lane/4 of the row goes to chunk position (lane/4) ^ (slot & 7)
            unsigned char *row = reinterpret_cast<unsigned char *>(p.k_pool) + (tile * kBS + slot) * kHD;
            reinterpret_cast<uint32_t *>(row + (((lane >> 2) ^ (slot & 7)) << 4))[lane & 3] = w;
            if (lane == 0) p.k_scale[tile * kBS + slot] = s;
        }
        // V row -> staged for the dim-major write
        {
            const float4 x = reinterpret_cast<const float4 *>(p.v_new + src)[lane];
            float m = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
            m = warp_max(m);
            const float s = kv_row_scale(m);
            v_stage[4 * lane + 0][r] = (int8_t)kv_code(x.x, s);
            v_stage[4 * lane + 1][r] = (int8_t)kv_code(x.y, s);
            v_stage[4 * lane + 2][r] = (int8_t)kv_code(x.z, s);
            v_stage[4 * lane + 3][r] = (int8_t)kv_code(x.w, s);
            if (lane == 0) p.v_scale[tile * kBS + slot] = s;
        }
    }
    __syncthreads();

    // Dim-major V write (per 64-token quarter): a warp stores one dim row for
    // the CTA's 32 tokens, which are consecutive slots except at a boundary.
    const int r = lane;
    const int phys = tok_phys[r];
    if (phys >= 0) {
        const int slot = tok_slot[r];
        const size_t base = ((size_t)phys * p.nkv + h) * kHD * kBS +
                            (size_t)(slot / kStageTok) * kTileVQuarter + (slot % kStageTok);
        for (int d = warp; d < kHD; d += kAppendWarps)
            p.v_pool[base + (size_t)d * kStageTok] = v_stage[d][r];
    }
}

// One new token per sequence (a decode step): a warp per (sequence, kv head),
// K row and V row quantised from one float4 per lane; no staging needed.
__global__ void __launch_bounds__(kAppendWarps * 32)
quantize_append_token_kernel(AppendParams p) {
    pdl_launch_dependents();  // let the next kernel of the step be scheduled now
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wid = blockIdx.x * kAppendWarps + warp;
    if (wid >= p.batch * p.nkv) return;
    const int b = wid / p.nkv, h = wid % p.nkv;
    const int cap = p.max_blocks * kBS;
    const int pos = start_position(p, b, cap);
    if (pos == kNoAppend) return;
    if (pos < 0 || pos >= cap) {
        if (lane == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_POSITION);
        return;
    }
    const int phys = p.block_table[(size_t)b * p.max_blocks + pos / kBS];
    if (phys < 0 || phys >= p.num_blocks) {
        if (lane == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_BLOCK_ID);
        return;
    }
    const int slot = pos % kBS;
    const size_t src = ((size_t)b * p.nkv + h) * kHD;   // n_new == 1
    const size_t tile = (size_t)phys * p.nkv + h;
    const float4 xk = reinterpret_cast<const float4 *>(p.k_new + src)[lane];
    const float4 xv = reinterpret_cast<const float4 *>(p.v_new + src)[lane];
    {
        const float m = warp_max(fmaxf(fmaxf(fabsf(xk.x), fabsf(xk.y)), fmaxf(fabsf(xk.z), fabsf(xk.w))));
        const float s = kv_row_scale(m);
        const uint32_t w = pack4(kv_code(xk.x, s), kv_code(xk.y, s), kv_code(xk.z, s), kv_code(xk.w, s));
        unsigned char *row = reinterpret_cast<unsigned char *>(p.k_pool) + (tile * kBS + slot) * kHD;
        reinterpret_cast<uint32_t *>(row + (((lane >> 2) ^ (slot & 7)) << 4))[lane & 3] = w;
        if (lane == 0) p.k_scale[tile * kBS + slot] = s;
    }
    {
        const float m = warp_max(fmaxf(fmaxf(fabsf(xv.x), fabsf(xv.y)), fmaxf(fabsf(xv.z), fabsf(xv.w))));
        const float s = kv_row_scale(m);
        int8_t *vg = p.v_pool + tile * kHD * kBS + (size_t)(slot / kStageTok) * kTileVQuarter + slot % kStageTok;
        vg[(size_t)(4 * lane + 0) * kStageTok] = (int8_t)kv_code(xv.x, s);
        vg[(size_t)(4 * lane + 1) * kStageTok] = (int8_t)kv_code(xv.y, s);
        vg[(size_t)(4 * lane + 2) * kStageTok] = (int8_t)kv_code(xv.z, s);
        vg[(size_t)(4 * lane + 3) * kStageTok] = (int8_t)kv_code(xv.w, s);
        if (lane == 0) p.v_scale[tile * kBS + slot] = s;
    }
}

__global__ void __launch_bounds__(128)
quantize_q_kernel(const float *__restrict__ q, int64_t n_rows, int8_t *__restrict__ codes,
                  float *__restrict__ scales) {
    const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (row >= n_rows) return;
    quantize_q_row_warp(q + row * kHD, threadIdx.x & 31, codes + row * kHD, scales + row * kNQB);
}

}  // namespace

cudaError_t launch_quantize_append(const AppendParams &p, cudaStream_t s) {
    if (p.n_new == 1) {
        const int64_t warps = (int64_t)p.batch * p.nkv;
        quantize_append_token_kernel<<<(unsigned)((warps + kAppendWarps - 1) / kAppendWarps),
                                       kAppendWarps * 32, 0, s>>>(p);
    } else {
        dim3 grid((p.n_new + kAppendTokens - 1) / kAppendTokens, p.nkv, p.batch);
        quantize_append_kernel<<<grid, kAppendWarps * 32, 0, s>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_quantize_q(const float *q, int64_t n_rows, int8_t *codes, float *scales,
                              cudaStream_t s) {
    const int64_t blocks = (n_rows + 3) / 4;
    quantize_q_kernel<<<(unsigned)blocks, 128, 0, s>>>(q, n_rows, codes, scales);
    return cudaGetLastError();
}

}  // namespace kvq8
