// f32.cu -- the fp32 KV cache ("mirror" cache): append and decode.
//
// [Day 9-1] §2-§3 keeps an fp32 copy of K/V next to the int8 cache, for
// debugging and comparison; [Day 9-3] §1 uses it as the baseline arm of its
// accuracy experiment.  Here it is a paged fp32 cache with the same tables:
//   k_cache, v_cache fp32 [num_blocks][nkv][256][hd]   token-major rows
// (1024 bytes per (token, kv head) for K and V together), and a decode that is
// plain softmax attention of the fp32 query over it, split over the context and
// merged by the same combine kernel as the q8 decode.
//
// Decode: one CTA per (split, kv head, sequence), 4 warps; a warp takes 8
// tokens at a time with all 16 row loads (K and V, one float4 per lane each) in
// flight, reduces the 8 x G dot products across the warp, updates its online
// softmax once per 8 tokens (one exponential per lane and head) and
// accumulates P.V with lane = 4 dims, the 8 weights broadcast through shared
// memory.
#include <math.h>

#include "kvq8_device.cuh"
#include "kvq8_internal.cuh"

namespace kvq8 {
namespace {

constexpr int kWarpsF = 4;
constexpr int kTokF = 8;          // tokens per warp step
constexpr int kChunkF = 64;       // tokens per warp chunk (walked kTokF at a time)

// One warp per new (token, kv head): copy the K and V rows into the cache.
__global__ void __launch_bounds__(256)
f32_append_kernel(F32AppendParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * 8 + warp, h = blockIdx.y, b = blockIdx.z;
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
    reinterpret_cast<float4 *>(p.k_cache + row * kHD)[lane] = reinterpret_cast<const float4 *>(p.k_new + src)[lane];
    reinterpret_cast<float4 *>(p.v_cache + row * kHD)[lane] = reinterpret_cast<const float4 *>(p.v_new + src)[lane];
}

// Sums a[j] (j < 8) over the warp's 32 lanes and returns, in lane l, the sum
// for j = l >> 2: at each of the first three steps a lane keeps the half of its
// values that its lane bit selects and adds the partner's copy of that half.
__device__ __forceinline__ float transpose_sum8(const float (&a)[kTokF], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float b[4], c[2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float keep = b4 ? a[j + 4] : a[j], send = b4 ? a[j] : a[j + 4];
        b[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float keep = b3 ? b[j + 2] : b[j], send = b3 ? b[j] : b[j + 2];
        c[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float d;
    {
        const float keep = b2 ? c[1] : c[0], send = b2 ? c[0] : c[1];
        d = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    d += __shfl_xor_sync(0xffffffffu, d, 2);
    d += __shfl_xor_sync(0xffffffffu, d, 1);
    return d;
}

template <int G>
__global__ void __launch_bounds__(kWarpsF * 32)
f32_decode_split_kernel(F32DecodeParams p) {
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
        const int nvalid = (L + p.split_tokens - 1) / p.split_tokens;
        p.ws_meta[u] = make_int2((int)(u * (p.nsplit - 1)), nvalid);
    }
    const int tok_begin = split * p.split_tokens;
    if (tok_begin >= L) return;
    const int tok_end = min(L, tok_begin + p.split_tokens);

    __shared__ float red_acc[kWarpsF][G][kHD];
    __shared__ __align__(16) float w_sm[kWarpsF][G][kTokF];
    __shared__ float red_ml[kWarpsF][G][2];

    // this lane's four dims of the G query heads, with the softmax scale folded in
    float4 qv[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float4 x = reinterpret_cast<const float4 *>(p.q + ((size_t)b * p.nqh + (size_t)h * G + g) * kHD)[lane];
        x.x *= p.sm_scale_log2; x.y *= p.sm_scale_log2; x.z *= p.sm_scale_log2; x.w *= p.sm_scale_log2;
        qv[g] = x;
    }
    float M[G], S[G];
    float4 acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        M[g] = -INFINITY;
        S[g] = 0.0f;
        acc[g] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    const int nchunks = (tok_end - tok_begin + kChunkF - 1) / kChunkF;
    for (int cidx = warp; cidx < nchunks; cidx += kWarpsF) {
        const int c0 = tok_begin + cidx * kChunkF;
        const int phys = p.block_table[(size_t)b * p.max_blocks + c0 / kBS];
        if (phys < 0 || phys >= p.num_blocks) {
            if (lane == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_BLOCK_ID);
            continue;
        }
        const size_t row0 = ((size_t)phys * p.nkv + h) * kBS + c0 % kBS;
        const int ntok = min(kChunkF, tok_end - c0);
        for (int t0 = 0; t0 < ntok; t0 += kTokF) {
            float4 kr[kTokF], vr[kTokF];
#pragma unroll
            for (int j = 0; j < kTokF; ++j) {
                if (t0 + j < ntok) {
                    kr[j] = reinterpret_cast<const float4 *>(p.k_cache + (row0 + t0 + j) * kHD)[lane];
                    vr[j] = reinterpret_cast<const float4 *>(p.v_cache + (row0 + t0 + j) * kHD)[lane];
                } else {
                    kr[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                    vr[j] = kr[j];
                }
            }
            // scores: the 8 x 32 partial dot products are summed by a
            // transposing butterfly that leaves lane l with the score of token
            // l >> 2 (9 shuffles for 8 tokens instead of 40)
            float alpha[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float a[kTokF];
#pragma unroll
                for (int j = 0; j < kTokF; ++j) {
                    float x = qv[g].x * kr[j].x;
                    x = fmaf(qv[g].y, kr[j].y, x);
                    x = fmaf(qv[g].z, kr[j].z, x);
                    a[j] = fmaf(qv[g].w, kr[j].w, x);
                }
                const float sc = transpose_sum8(a, lane);
                const float sv = (t0 + (lane >> 2) < ntok) ? sc : -INFINITY;
                float m = fmaxf(sv, __shfl_xor_sync(0xffffffffu, sv, 4));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                const float m_new = fmaxf(M[g], m);   // finite: token t0 is valid
                alpha[g] = exp2f(M[g] - m_new);
                M[g] = m_new;
                const float w = exp2f(sv - m_new);    // 0 for tokens past the end
                S[g] = fmaf(S[g], alpha[g], w);       // per lane: its token's weights
                if ((lane & 3) == 0) w_sm[warp][g][lane >> 2] = w;
            }
            __syncwarp();
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float4 w0 = reinterpret_cast<const float4 *>(w_sm[warp][g])[0];
                const float4 w1 = reinterpret_cast<const float4 *>(w_sm[warp][g])[1];
                const float wj[kTokF] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                float4 a4 = make_float4(acc[g].x * alpha[g], acc[g].y * alpha[g],
                                        acc[g].z * alpha[g], acc[g].w * alpha[g]);
#pragma unroll
                for (int j = 0; j < kTokF; ++j) {
                    a4.x = fmaf(wj[j], vr[j].x, a4.x);
                    a4.y = fmaf(wj[j], vr[j].y, a4.y);
                    a4.z = fmaf(wj[j], vr[j].z, a4.z);
                    a4.w = fmaf(wj[j], vr[j].w, a4.w);
                }
                acc[g] = a4;
            }
            __syncwarp();
        }
    }
    // a lane's S holds the weights of one token class; the 8 classes sit in
    // lanes that differ in bits 2..4 (the four copies in bits 0..1 are equal)
#pragma unroll
    for (int g = 0; g < G; ++g) {
        S[g] += __shfl_xor_sync(0xffffffffu, S[g], 4);
        S[g] += __shfl_xor_sync(0xffffffffu, S[g], 8);
        S[g] += __shfl_xor_sync(0xffffffffu, S[g], 16);
    }

    // merge the warps' states into one record per query head
#pragma unroll
    for (int g = 0; g < G; ++g) {
        reinterpret_cast<float4 *>(red_acc[warp][g])[lane] = acc[g];
        if (lane == 0) {
            red_ml[warp][g][0] = M[g];
            red_ml[warp][g][1] = S[g];
        }
    }
    __syncthreads();
    const int d = threadIdx.x;
    const size_t rec = u * p.nsplit + split;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float m = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarpsF; ++w) m = fmaxf(m, red_ml[w][g][0]);
        float s_sum = 0.0f, a = 0.0f;
        if (m != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarpsF; ++w) {
                const float f = exp2f(red_ml[w][g][0] - m);
                s_sum = fmaf(red_ml[w][g][1], f, s_sum);
                a = fmaf(red_acc[w][g][d], f, a);
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

// Splits per (sequence, kv head) so that the grid holds about 8 CTAs per SM
// (152 SMs), each split a whole number of 64-token chunks.
bool make_f32_plan(int batch, int nkv, int max_blocks, int *nsplit, int *split_tokens) {
    const int64_t units = (int64_t)batch * nkv;
    if (units <= 0 || max_blocks <= 0) return false;
    const int64_t cap_tokens = (int64_t)max_blocks * kBS;
    int64_t ns = (152 * 8 + units - 1) / units;
    ns = ns < 1 ? 1 : ns;
    ns = ns > 1 + kMaxCtas / units ? 1 + kMaxCtas / units : ns;
    int64_t st = (cap_tokens + ns - 1) / ns;
    st = (st + kChunkF - 1) / kChunkF * kChunkF;
    *split_tokens = (int)st;
    *nsplit = (int)((cap_tokens + st - 1) / st);
    return true;
}

cudaError_t launch_f32_append(const F32AppendParams &p, cudaStream_t s) {
    dim3 grid((p.n_new + 7) / 8, p.nkv, p.batch);
    f32_append_kernel<<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_f32_decode_split(const F32DecodeParams &p, int group, cudaStream_t s) {
    dim3 grid(p.nsplit, p.nkv, p.batch);
    switch (group) {
        case 1: f32_decode_split_kernel<1><<<grid, kWarpsF * 32, 0, s>>>(p); break;
        case 2: f32_decode_split_kernel<2><<<grid, kWarpsF * 32, 0, s>>>(p); break;
        case 4: f32_decode_split_kernel<4><<<grid, kWarpsF * 32, 0, s>>>(p); break;
        case 8: f32_decode_split_kernel<8><<<grid, kWarpsF * 32, 0, s>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace kvq8
