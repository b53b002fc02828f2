// int4.cu -- the asymmetric INT4 group-64 KV cache: quantise-append and the
// split-KV decode over it.
//
// Rule ([UltraQuant] §3.2 code): per group of 64 consecutive values of a
// (token, kv head) row, scale = (max - min)/15 (1 when max == min),
// zero = round_half_even(-min/scale) kept in fp32, code = clamp(round_half_even
// (x/scale + zero), 0, 15); two codes per byte, the even element in the high
// nibble; dequantised value (code - zero) * scale.  Decode takes the fp32
// query against the dequantised K/V (the page dequantises and runs standard
// attention).
//
// Cache layout (per (block, kv head) tile of 256 tokens):
//   codes  uint8 [256][64]   token-major, byte i = code[2i] << 4 | code[2i+1]
//   params fp32  [256][4]    (scale of dims 0-63, its zero, scale of 64-127, its zero)
// for K and for V: 160 bytes per (token, kv head).
//
// Decode: one CTA per (split, kv head, sequence), 4 warps walking the split in
// 32-token chunks, each warp with its own online-softmax state.  Lane = token
// for Q.K: s = sm_scale * sum_g scale_g * (sum_{d in g} q_d c_d - zero_g *
// sum_{d in g} q_d), i.e. exactly q . dequant(k); lane = 4 dims for P.V.  The
// warps' states are merged into one partial record per query head, in the
// record format of the q8 decode, so the same combine kernel finishes it.
#include <math.h>

#include "kvq8_device.cuh"
#include "kvq8_internal.cuh"
#include "kvq8_ptx.cuh"

namespace kvq8 {
namespace {

constexpr int kRowBytes = kHD / 2;          // 64 bytes of codes per (token, head)
constexpr int kAppendWarps4 = 8;
constexpr int kWarps4 = 4;
constexpr int kChunk4 = 32;
constexpr int kKRow4 = kRowBytes + 16;      // padded K row in shared memory

// 16 lanes (a half warp) reduce one 64-value group.
__device__ __forceinline__ float half_max(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float half_min(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ int int4_code(float x, float s, float z) {
    const int c = __float2int_rn(__fadd_rn(__fdiv_rn(x, s), z));
    return max(0, min(15, c));
}

// Quantises one row (lane l holds dims 4l..4l+3) and stores codes + params.
__device__ __forceinline__ void int4_store_row(const float4 x, uint8_t *codes_row, float *param_row,
                                               int lane) {
    float mx = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
    float mn = fminf(fminf(x.x, x.y), fminf(x.z, x.w));
    mx = half_max(mx);
    mn = half_min(mn);
    const float s = (mx != mn) ? __fdiv_rn(__fsub_rn(mx, mn), 15.0f) : 1.0f;
    const float z = rintf(__fdiv_rn(-mn, s));
    const int c0 = int4_code(x.x, s, z), c1 = int4_code(x.y, s, z);
    const int c2 = int4_code(x.z, s, z), c3 = int4_code(x.w, s, z);
    const uint16_t two = (uint16_t)(((c0 << 4) | c1) | (((c2 << 4) | c3) << 8));
    reinterpret_cast<uint16_t *>(codes_row)[lane] = two;
    if ((lane & 15) == 0) {
        param_row[(lane >> 4) * 2 + 0] = s;
        param_row[(lane >> 4) * 2 + 1] = z;
    }
}

// One warp per new (token, kv head): K row then V row.
__global__ void __launch_bounds__(kAppendWarps4 * 32)
int4_append_kernel(Int4AppendParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * kAppendWarps4 + warp, h = blockIdx.y, b = blockIdx.z;
    if (i >= p.n_new) return;
    const int cap = p.max_blocks * kBS;
    const int pos = p.start_pos[b] + i;
    if (pos < 0 || pos >= cap) {
        if (lane == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_POSITION);
        return;
    }
    const int phys = p.block_table[(size_t)b * p.max_blocks + pos / kBS];
    if (phys < 0 || phys >= p.num_blocks) {
        if (lane == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_BLOCK_ID);
        return;
    }
    const size_t row = ((size_t)phys * p.nkv + h) * kBS + pos % kBS;
    const size_t src = (((size_t)b * p.n_new + i) * p.nkv + h) * kHD;
    int4_store_row(reinterpret_cast<const float4 *>(p.k_new + src)[lane], p.k_codes + row * kRowBytes,
                   p.k_param + row * 4, lane);
    int4_store_row(reinterpret_cast<const float4 *>(p.v_new + src)[lane], p.v_codes + row * kRowBytes,
                   p.v_param + row * 4, lane);
}

template <int G>
struct Int4Smem {
    float q[G][kHD];
    float qsum[G][2];
    union {
        struct {
            uint8_t k[kWarps4][kChunk4][kKRow4];
            uint8_t v[kWarps4][kChunk4][kRowBytes];
            float4 kp[kWarps4][kChunk4];
            float4 vp[kWarps4][kChunk4];
            float pw[kWarps4][kChunk4][G];
        } loop;
        float red_acc[kWarps4][G][kHD];
    } u;
    float red_ml[kWarps4][G][2];
};

__device__ __forceinline__ float nib(uint32_t w, int shift) { return (float)((w >> shift) & 0xFu); }

template <int G>
__global__ void __launch_bounds__(kWarps4 * 32)
int4_decode_split_kernel(Int4DecodeParams p) {
    pdl_wait();
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cap = p.max_blocks * kBS;
    int L = p.ctx_lens[b];
    if (L < 0 || L > cap) {
        if (threadIdx.x == 0 && split == 0 && h == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_CTX_LEN);
        L = max(0, min(L, cap));
    }
    const size_t u = (size_t)b * p.nkv + h;
    if (split == 0 && threadIdx.x == 0) {
        // records of unit u are u*nsplit + j; the combine reads first + u + j
        const int nvalid = (L + p.split_tokens - 1) / p.split_tokens;
        p.ws_meta[u] = make_int2((int)(u * (p.nsplit - 1)), nvalid);
    }
    const int tok_begin = split * p.split_tokens;
    if (tok_begin >= L) return;
    const int tok_end = min(L, tok_begin + p.split_tokens);

    __shared__ __align__(16) Int4Smem<G> sm;
    for (int i = threadIdx.x; i < G * kHD; i += kWarps4 * 32)
        sm.q[i / kHD][i % kHD] = p.q[((size_t)b * p.nqh + (size_t)h * G) * kHD + i];
    __syncthreads();
    if (threadIdx.x < 2 * G) {
        const int g = threadIdx.x >> 1, grp = threadIdx.x & 1;
        float s = 0.0f;
        for (int d = 0; d < 64; ++d) s += sm.q[g][grp * 64 + d];
        sm.qsum[g][grp] = s;
    }
    __syncthreads();

    float M[G], S[G], acc[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        M[g] = -INFINITY;
        S[g] = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[g][j] = 0.0f;
    }
    const int vgrp = lane >> 4;  // group of this lane's four V dims

    const int nchunks = (tok_end - tok_begin + kChunk4 - 1) / kChunk4;
    for (int cidx = warp; cidx < nchunks; cidx += kWarps4) {
        const int t0 = tok_begin + cidx * kChunk4;
        const int phys = p.block_table[(size_t)b * p.max_blocks + t0 / kBS];
        if (phys < 0 || phys >= p.num_blocks) {
            if (lane == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_BLOCK_ID);
            continue;
        }
        const size_t row0 = ((size_t)phys * p.nkv + h) * kBS + t0 % kBS;
        // stage 32 K rows, 32 V rows (16-byte loads, coalesced) and their params
        const uint8_t *kg = p.k_codes + row0 * kRowBytes;
        const uint8_t *vg = p.v_codes + row0 * kRowBytes;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int r = it * 8 + (lane >> 2), ch = lane & 3;
            *reinterpret_cast<int4 *>(&sm.u.loop.k[warp][r][ch * 16]) =
                *reinterpret_cast<const int4 *>(kg + r * kRowBytes + ch * 16);
            *reinterpret_cast<int4 *>(&sm.u.loop.v[warp][r][ch * 16]) =
                *reinterpret_cast<const int4 *>(vg + r * kRowBytes + ch * 16);
        }
        sm.u.loop.kp[warp][lane] = reinterpret_cast<const float4 *>(p.k_param)[row0 + lane];
        sm.u.loop.vp[warp][lane] = reinterpret_cast<const float4 *>(p.v_param)[row0 + lane];
        __syncwarp();

        // Q.K, lane = token
        const bool valid = t0 + lane < tok_end;
        float dot[G][2];
#pragma unroll
        for (int g = 0; g < G; ++g) dot[g][0] = dot[g][1] = 0.0f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const int4 kw = *reinterpret_cast<const int4 *>(&sm.u.loop.k[warp][lane][cc * 16]);
            const uint32_t words[4] = {(uint32_t)kw.x, (uint32_t)kw.y, (uint32_t)kw.z, (uint32_t)kw.w};
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
                // 8 dims: byte k holds dims 2k (high nibble) and 2k+1 (low)
                const uint32_t w = words[wi];
                const float c[8] = {nib(w, 4), nib(w, 0), nib(w, 12), nib(w, 8),
                                    nib(w, 20), nib(w, 16), nib(w, 28), nib(w, 24)};
                const int d0 = cc * 32 + wi * 8;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float4 qa = *reinterpret_cast<const float4 *>(&sm.q[g][d0]);
                    const float4 qb = *reinterpret_cast<const float4 *>(&sm.q[g][d0 + 4]);
                    float a = dot[g][cc >> 1];
                    a = fmaf(qa.x, c[0], a); a = fmaf(qa.y, c[1], a);
                    a = fmaf(qa.z, c[2], a); a = fmaf(qa.w, c[3], a);
                    a = fmaf(qb.x, c[4], a); a = fmaf(qb.y, c[5], a);
                    a = fmaf(qb.z, c[6], a); a = fmaf(qb.w, c[7], a);
                    dot[g][cc >> 1] = a;
                }
            }
        }
        const float4 kp = sm.u.loop.kp[warp][lane];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float s = -INFINITY;
            if (valid) {
                const float a0 = kp.x * (dot[g][0] - kp.y * sm.qsum[g][0]);
                const float a1 = kp.z * (dot[g][1] - kp.w * sm.qsum[g][1]);
                s = (a0 + a1) * p.sm_scale_log2;
            }
            const float m_new = fmaxf(M[g], warp_max(s));  // finite: token t0 is valid
            const float alpha = exp2f(M[g] - m_new);
            const float w = valid ? exp2f(s - m_new) : 0.0f;
            S[g] = S[g] * alpha + warp_sum(w);
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[g][j] *= alpha;
            M[g] = m_new;
            sm.u.loop.pw[warp][lane][g] = w;
        }
        __syncwarp();

        // P.V, lane = dims 4l..4l+3 (bytes 2l, 2l+1 of each V row)
        const int ntok = min(kChunk4, tok_end - t0);
        for (int t = 0; t < ntok; ++t) {
            const uint32_t two = reinterpret_cast<const uint16_t *>(&sm.u.loop.v[warp][t][0])[lane];
            const float4 vp = sm.u.loop.vp[warp][t];
            const float vs = vgrp ? vp.z : vp.x, vz = vgrp ? vp.w : vp.y;
            const float v0 = (nib(two, 4) - vz) * vs, v1 = (nib(two, 0) - vz) * vs;
            const float v2 = (nib(two, 12) - vz) * vs, v3 = (nib(two, 8) - vz) * vs;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float pw = sm.u.loop.pw[warp][t][g];
                acc[g][0] = fmaf(pw, v0, acc[g][0]);
                acc[g][1] = fmaf(pw, v1, acc[g][1]);
                acc[g][2] = fmaf(pw, v2, acc[g][2]);
                acc[g][3] = fmaf(pw, v3, acc[g][3]);
            }
        }
        __syncwarp();
    }

    // merge the warps' states into one record per query head
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int j = 0; j < 4; ++j) sm.u.red_acc[warp][g][4 * lane + j] = acc[g][j];
        if (lane == 0) {
            sm.red_ml[warp][g][0] = M[g];
            sm.red_ml[warp][g][1] = S[g];
        }
    }
    __syncthreads();
    const int d = threadIdx.x;
    const size_t rec = u * p.nsplit + split;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float m = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps4; ++w) m = fmaxf(m, sm.red_ml[w][g][0]);
        float s_sum = 0.0f, a = 0.0f;
        if (m != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps4; ++w) {
                const float f = exp2f(sm.red_ml[w][g][0] - m);
                s_sum = fmaf(sm.red_ml[w][g][1], f, s_sum);
                a = fmaf(sm.u.red_acc[w][g][d], f, a);
            }
        }
        p.ws_acc[(rec * G + g) * kHD + d] = a;
        if (d == 0) {
            p.ws_ml[(rec * G + g) * 2 + 0] = m;
            p.ws_ml[(rec * G + g) * 2 + 1] = s_sum;
        }
    }
}

}  // namespace

// Splits: enough CTAs for several waves, within the record budget of the
// decode workspace (kMaxCtas + units records).
bool make_int4_plan(int batch, int nkv, int max_blocks, int *nsplit, int *split_tokens) {
    const int64_t units = (int64_t)batch * nkv;
    if (units <= 0 || max_blocks <= 0) return false;
    const int64_t cap_tokens = (int64_t)max_blocks * kBS;
    int64_t ns = (152 * 8 + units - 1) / units;
    ns = ns < 1 ? 1 : ns;
    ns = ns > 1 + kMaxCtas / units ? 1 + kMaxCtas / units : ns;
    int64_t st = (cap_tokens + ns - 1) / ns;
    st = (st + kChunk4 - 1) / kChunk4 * kChunk4;
    *split_tokens = (int)st;
    *nsplit = (int)((cap_tokens + st - 1) / st);
    return true;
}

cudaError_t launch_int4_append(const Int4AppendParams &p, cudaStream_t s) {
    dim3 grid((p.n_new + kAppendWarps4 - 1) / kAppendWarps4, p.nkv, p.batch);
    int4_append_kernel<<<grid, kAppendWarps4 * 32, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_int4_decode_split(const Int4DecodeParams &p, int group, cudaStream_t s) {
    dim3 grid(p.nsplit, p.nkv, p.batch);
    switch (group) {
        case 1: int4_decode_split_kernel<1><<<grid, kWarps4 * 32, 0, s>>>(p); break;
        case 2: int4_decode_split_kernel<2><<<grid, kWarps4 * 32, 0, s>>>(p); break;
        case 4: int4_decode_split_kernel<4><<<grid, kWarps4 * 32, 0, s>>>(p); break;
        case 8: int4_decode_split_kernel<8><<<grid, kWarps4 * 32, 0, s>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace kvq8
