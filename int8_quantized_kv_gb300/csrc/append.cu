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

constexpr int kAppendWarps = 8;                  // one-token kernel: warps per CTA
constexpr int kQWarps = 16;                      // quarter kernel: warps per CTA
constexpr int kQTok = kStageTok;                 // tokens per CTA: one 64-token quarter
constexpr int kRowsPerWarp = kQTok / kQWarps;
constexpr int kVStride = kQTok + 4;              // staged V dim row: 17 words, conflict-free
constexpr int kNoAppend = INT_MIN;               // this sequence appends nothing

// kv_code of four values of one row whose scale is sc = fl(max|row| / 127),
// with one reciprocal per row in place of a division per value.  For |v| <=
// max|row|, |v / sc| < 127.0001; p = fl(v * fl(1 / sc)) carries two roundings,
// so |p - v / sc| < 127.0001 * (2^-23 + 2^-46) < 2^-16, and fl(v / sc) lies
// within half an ulp below 128 (2^-18) of v / sc: |p - fl(v / sc)| < 2^-15.
// Where p is at least 2^-15 from every half-integer, p and fl(v / sc) round
// to the same integer (|p| < 127.5, so no clamp is needed); the four values
// are divided exactly when one of them is closer (about 6e-5 of values) or
// when sc lies outside [2^-120, 2^120] (a zero row, a subnormal or non-finite
// scale), which gives kv_code's result in every case.
__device__ __forceinline__ int4 kv_codes4(float4 x, float sc) {
    if (sc >= 0x1p-120f && sc <= 0x1p120f) {
        const float inv = __frcp_rn(sc);
        const float p0 = __fmul_rn(x.x, inv), p1 = __fmul_rn(x.y, inv);
        const float p2 = __fmul_rn(x.z, inv), p3 = __fmul_rn(x.w, inv);
        const float r0 = rintf(p0), r1 = rintf(p1), r2 = rintf(p2), r3 = rintf(p3);
        constexpr float kLim = 0.5f - 0x1p-15f;
        const float d = fmaxf(fmaxf(fabsf(p0 - r0), fabsf(p1 - r1)),
                              fmaxf(fabsf(p2 - r2), fabsf(p3 - r3)));
        if (d <= kLim)
            return make_int4(__float2int_rn(r0), __float2int_rn(r1), __float2int_rn(r2),
                             __float2int_rn(r3));
    }
    return make_int4(kv_code(x.x, sc), kv_code(x.y, sc), kv_code(x.z, sc), kv_code(x.w, sc));
}

// Position of the first new token of sequence b: start_pos[b], or in a decode
// step ctx_lens[b] - 1 (nothing for an empty or out-of-table context, which
// the decode flags).
__device__ __forceinline__ int start_position(const AppendParams &p, int b, int cap) {
    if (p.start_pos) return p.start_pos[b];
    const int L = p.ctx_lens[b];
    return (L >= 1 && L <= cap) ? L - 1 : kNoAppend;
}

// One CTA per 64-token quarter of the cache touched by the new tokens of one
// (sequence, kv head): CTA x takes quarter floor(start/64) + x.  Every warp
// first issues the loads of its 4 rows (K and V), then quantises them; K rows
// go to the token-major tile, V codes through shared memory to the dim-major
// quarter, which a full quarter writes as one contiguous 8 KiB run.
__global__ void __launch_bounds__(kQWarps * 32)
quantize_append_kernel(AppendParams p) {
    const int h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    __shared__ __align__(16) int8_t v_stage[kHD][kVStride];
    __shared__ __align__(16) float v_sc[kQTok];

    pdl_launch_dependents();  // let the next kernel of the step be scheduled now
    const int cap = p.max_blocks * kBS;
    const int start = start_position(p, b, cap);
    if (start == kNoAppend) return;
    const long long q0 = ((long long)start >= 0 ? start / kQTok : -(((long long)-start + kQTok - 1) / kQTok));
    const long long qpos = (q0 + blockIdx.x) * kQTok;          // first position of this quarter
    const long long lo = max((long long)start, qpos);
    const long long hi = min((long long)start + p.n_new, qpos + kQTok);
    if (lo >= hi) return;                                        // block-uniform
    if (lo < 0 || hi > cap) {
        if (threadIdx.x == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_POSITION);
        if (hi <= 0 || lo >= cap) return;
    }
    const long long vlo = max(lo, 0LL), vhi = min(hi, (long long)cap);  // positions inside the table
    const int phys = p.block_table[(size_t)b * p.max_blocks + (int)(qpos / kBS)];
    if (phys < 0 || phys >= p.num_blocks) {
        if (threadIdx.x == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_BLOCK_ID);
        return;
    }
    const size_t tile = (size_t)phys * p.nkv + h;
    const int slot0 = (int)(qpos % kBS);                         // first slot of the quarter

    // this warp's rows: quarter offsets r = warp + 16j.  K: lane l holds dims
    // 4l..4l+3 (one packed word of codes); V: lane l holds dims l + 32k, so that
    // the transposing writes below hit 32 different banks
    float4 xk[kRowsPerWarp], xv[kRowsPerWarp];
#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j) {
        const long long pos = qpos + warp + kQWarps * j;
        if (pos >= vlo && pos < vhi) {
            const size_t src = (((size_t)b * p.n_new + (size_t)(pos - start)) * p.nkv + h) * kHD;
            xk[j] = reinterpret_cast<const float4 *>(p.k_new + src)[lane];
            const float *vr = p.v_new + src;
            xv[j] = make_float4(vr[lane], vr[lane + 32], vr[lane + 64], vr[lane + 96]);
        }
    }
#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j) {
        const int r = warp + kQWarps * j;
        const long long pos = qpos + r;
        if (pos < vlo || pos >= vhi) continue;                   // warp-uniform
        const int slot = slot0 + r;
        {
            const float4 x = xk[j];
            float m = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
            m = warp_max(m);
            const float sc = kv_row_scale(m);
            const int4 c = kv_codes4(x, sc);
            const uint32_t w = pack4(c.x, c.y, c.z, c.w);
            // 16-byte chunk lane/4 of the row goes to chunk position (lane/4) ^ (slot & 7)
            unsigned char *row = reinterpret_cast<unsigned char *>(p.k_pool) + (tile * kBS + slot) * kHD;
            reinterpret_cast<uint32_t *>(row + (((lane >> 2) ^ (slot & 7)) << 4))[lane & 3] = w;
            if (lane == 0) p.k_scale[tile * kBS + slot] = sc;
        }
        {
            const float4 x = xv[j];
            float m = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
            m = warp_max(m);
            const float sc = kv_row_scale(m);
            const int4 c = kv_codes4(x, sc);
            v_stage[lane + 0][r] = (int8_t)c.x;
            v_stage[lane + 32][r] = (int8_t)c.y;
            v_stage[lane + 64][r] = (int8_t)c.z;
            v_stage[lane + 96][r] = (int8_t)c.w;
            if (lane == 0) v_sc[r] = sc;
        }
    }
    __syncthreads();

    int8_t *vq = p.v_pool + tile * kHD * kBS + (size_t)(slot0 / kQTok) * kTileVQuarter;
    if (vlo == qpos && vhi == qpos + kQTok) {
        // the whole quarter: 128 dim rows of 64 bytes, one 8 KiB run, 16-byte stores
        for (int e = threadIdx.x; e < kHD * (kQTok / 16); e += kQWarps * 32) {
            const int d = e / (kQTok / 16), c16 = e % (kQTok / 16);
            const uint32_t *w = reinterpret_cast<const uint32_t *>(&v_stage[d][16 * c16]);
            reinterpret_cast<int4 *>(vq + (size_t)d * kQTok)[c16] =
                make_int4((int)w[0], (int)w[1], (int)w[2], (int)w[3]);
        }
        if (threadIdx.x < kQTok / 4)
            reinterpret_cast<float4 *>(p.v_scale + tile * kBS + slot0)[threadIdx.x] =
                reinterpret_cast<const float4 *>(v_sc)[threadIdx.x];
    } else {
        // part of a quarter: one byte per (dim, new token)
        const int r0 = (int)(vlo - qpos), r1 = (int)(vhi - qpos);
        for (int e = threadIdx.x; e < kHD * kQTok; e += kQWarps * 32) {
            const int d = e / kQTok, r = e % kQTok;
            if (r >= r0 && r < r1) vq[(size_t)d * kQTok + r] = v_stage[d][r];
        }
        if (threadIdx.x >= r0 && threadIdx.x < r1) p.v_scale[tile * kBS + slot0 + threadIdx.x] = v_sc[threadIdx.x];
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
        const int4 c = kv_codes4(xk, s);
        const uint32_t w = pack4(c.x, c.y, c.z, c.w);
        unsigned char *row = reinterpret_cast<unsigned char *>(p.k_pool) + (tile * kBS + slot) * kHD;
        reinterpret_cast<uint32_t *>(row + (((lane >> 2) ^ (slot & 7)) << 4))[lane & 3] = w;
        if (lane == 0) p.k_scale[tile * kBS + slot] = s;
    }
    {
        const float m = warp_max(fmaxf(fmaxf(fabsf(xv.x), fabsf(xv.y)), fmaxf(fabsf(xv.z), fabsf(xv.w))));
        const float s = kv_row_scale(m);
        int8_t *vg = p.v_pool + tile * kHD * kBS + (size_t)(slot / kStageTok) * kTileVQuarter + slot % kStageTok;
        const int4 c = kv_codes4(xv, s);
        vg[(size_t)(4 * lane + 0) * kStageTok] = (int8_t)c.x;
        vg[(size_t)(4 * lane + 1) * kStageTok] = (int8_t)c.y;
        vg[(size_t)(4 * lane + 2) * kStageTok] = (int8_t)c.z;
        vg[(size_t)(4 * lane + 3) * kStageTok] = (int8_t)c.w;
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
        // quarters touched by n_new consecutive positions: at most n_new/64 + 1
        dim3 grid(p.n_new / kQTok + (p.n_new % kQTok ? 2 : 1), p.nkv, p.batch);
        quantize_append_kernel<<<grid, kQWarps * 32, 0, s>>>(p);
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
