// decode.cu -- split-KV single-query decode attention over the paged INT8
// cache, and the merge of the split results.
//
// Method: [Day 9-2] "flash_attn_single_q_q8_neon" §1-§3.  The query heads that
// share a kv head are quantised once in 32-blocks (segment 1); every cached
// token's score is rebuilt from exact int32 block dots times the query block
// scales, times the token's K scale and the softmax scale (segment 2, "three
// key points"); the softmax runs online with a running maximum, rescaling the
// running sum and the V accumulator when the maximum grows; V enters as int8
// code * (weight * V scale) in fp32; one division by the sum at the end
// (segment 3).
//
// GB300 layout of the work: one CTA = (split of a unit, kv head, sequence); its
// 4 warps walk the split in 32-token chunks, each warp with its own online
// softmax state.  Inside a chunk, lane t scores token t for all G query heads
// (dp4a over the K row staged in shared memory) and then the warp accumulates
// P.V with lane l owning dims l, l+32, l+64, l+96.  The 4 warp states are
// merged in shared memory into one partial record per query head; a second
// kernel merges the records of all splits and divides by the sum.
// The softmax runs in base 2: scores are pre-multiplied by log2(e), which
// leaves the normalised weights unchanged.
#include <math.h>

#include "kvq8_device.cuh"
#include "kvq8_internal.cuh"

namespace kvq8 {
namespace {

constexpr int kWarps = 4;
constexpr int kChunk = 32;            // tokens per warp iteration
constexpr int kKRow = kHD + 16;       // padded K row in shared memory (bytes)
constexpr int kVRow = kChunk + 4;     // padded V dim row in shared memory (bytes)

template <int G>
struct SplitSmem {
    int8_t q_codes[G][kHD];
    float q_scale[G][kNQB];
    union {
        struct {
            int8_t k_tile[kWarps][kChunk][kKRow];
            int8_t v_tile[kWarps][kHD][kVRow];
            float p[kWarps][kChunk][G];
        } loop;
        float red_acc[kWarps][G][kHD];
    } u;
    float red_ml[kWarps][G][2];
};

template <int G>
__global__ void __launch_bounds__(kWarps * 32)
decode_split_kernel(DecodeParams p) {
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int cap = p.max_blocks * kBS;
    int L = p.ctx_lens[b];
    if (L < 0 || L > cap) {
        if (threadIdx.x == 0 && split == 0 && h == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_CTX_LEN);
        L = max(0, min(L, cap));
    }
    const int tok_begin = split * p.split_blocks * kBS;
    if (tok_begin >= L) return;  // this split is empty; combine does not read its record
    const int tok_end = min(L, tok_begin + p.split_blocks * kBS);

    __shared__ __align__(16) SplitSmem<G> sm;

    // segment 1: quantise the G query heads of this kv head once
    for (int g = warp; g < G; g += kWarps)
        quantize_q_row_warp(p.q + ((size_t)b * p.nqh + (size_t)h * G + g) * kHD, lane,
                            sm.q_codes[g], sm.q_scale[g]);
    __syncthreads();

    float M[G], S[G], acc[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        M[g] = -INFINITY;
        S[g] = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[g][j] = 0.0f;
    }

    const int nchunks = (tok_end - tok_begin + kChunk - 1) / kChunk;
    for (int c = warp; c < nchunks; c += kWarps) {
        const int t0 = tok_begin + c * kChunk;
        const int slot0 = t0 % kBS;
        const int phys = p.block_table[(size_t)b * p.max_blocks + t0 / kBS];
        if (phys < 0 || phys >= p.num_blocks) {  // warp-uniform
            if (lane == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_BLOCK_ID);
            continue;
        }
        const size_t tile = (size_t)phys * p.nkv + h;

        // stage the chunk's 32 K rows and the V dim rows (coalesced 16-byte loads)
        const int8_t *kg = p.k_pool + (tile * kBS + slot0) * kHD;
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int row = it * 4 + (lane >> 3), ch = lane & 7;
            const int4 v = *reinterpret_cast<const int4 *>(kg + row * kHD + ch * 16);
            *reinterpret_cast<int4 *>(&sm.u.loop.k_tile[warp][row][ch * 16]) = v;
        }
        const int8_t *vg = p.v_pool + tile * kHD * kBS + slot0;
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int e = it * 32 + lane, d = e >> 1, half = e & 1;
            const int4 v = *reinterpret_cast<const int4 *>(vg + (size_t)d * kBS + half * 16);
            int *dst = reinterpret_cast<int *>(&sm.u.loop.v_tile[warp][d][half * 16]);
            dst[0] = v.x;
            dst[1] = v.y;
            dst[2] = v.z;
            dst[3] = v.w;
        }
        const bool valid = (t0 + lane) < tok_end;
        const float ks = p.k_scale[tile * kBS + slot0 + lane];
        const float vs = p.v_scale[tile * kBS + slot0 + lane];
        __syncwarp();

        // segment 2a: integer block dots, lane = token
        int dot[G][kNQB];
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int k = 0; k < kNQB; ++k) dot[g][k] = 0;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
            const int4 kw = *reinterpret_cast<const int4 *>(&sm.u.loop.k_tile[warp][lane][cc * 16]);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const int4 qw = *reinterpret_cast<const int4 *>(&sm.q_codes[g][cc * 16]);
                int d = dot[g][cc >> 1];
                d = __dp4a(kw.x, qw.x, d);
                d = __dp4a(kw.y, qw.y, d);
                d = __dp4a(kw.z, qw.z, d);
                d = __dp4a(kw.w, qw.w, d);
                dot[g][cc >> 1] = d;
            }
        }

        // segment 2b: scales, online softmax (one rescale per chunk)
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float s = -INFINITY;
            if (valid) {
                float a = (float)dot[g][0] * sm.q_scale[g][0];
#pragma unroll
                for (int k = 1; k < kNQB; ++k) a += (float)dot[g][k] * sm.q_scale[g][k];
                s = a * ks * p.sm_scale_log2;
            }
            const float m_new = fmaxf(M[g], warp_max(s));  // finite: lane 0 is valid
            const float alpha = exp2f(M[g] - m_new);       // 0 while M is -inf
            const float w = valid ? exp2f(s - m_new) : 0.0f;
            S[g] = S[g] * alpha + warp_sum(w);
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[g][j] *= alpha;
            M[g] = m_new;
            sm.u.loop.p[warp][lane][g] = valid ? w * vs : 0.0f;
        }
        __syncwarp();

        // segment 2c: acc += int8 V * (weight * V scale), lane = dims
#pragma unroll
        for (int wi = 0; wi < kChunk / 4; ++wi) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int word = *reinterpret_cast<const int *>(&sm.u.loop.v_tile[warp][lane + 32 * j][wi * 4]);
#pragma unroll
                for (int tt = 0; tt < 4; ++tt) {
                    const float v = (float)(int8_t)(word >> (8 * tt));
#pragma unroll
                    for (int g = 0; g < G; ++g) acc[g][j] += sm.u.loop.p[warp][wi * 4 + tt][g] * v;
                }
            }
        }
        __syncwarp();
    }

    // merge the 4 warp states into one record per query head
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int j = 0; j < 4; ++j) sm.u.red_acc[warp][g][lane + 32 * j] = acc[g][j];
        if (lane == 0) {
            sm.red_ml[warp][g][0] = M[g];
            sm.red_ml[warp][g][1] = S[g];
        }
    }
    __syncthreads();
    const int i = threadIdx.x;  // one dim per thread
    const size_t rec = ((size_t)b * p.nkv + h) * p.nsplit + split;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float m = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) m = fmaxf(m, sm.red_ml[w][g][0]);
        float s_sum = 0.0f, a = 0.0f;
        if (m != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = exp2f(sm.red_ml[w][g][0] - m);
                s_sum += sm.red_ml[w][g][1] * f;
                a += sm.u.red_acc[w][g][i] * f;
            }
        }
        p.ws_acc[(rec * G + g) * kHD + i] = a;
        if (i == 0) {
            p.ws_ml[(rec * G + g) * 2 + 0] = m;
            p.ws_ml[(rec * G + g) * 2 + 1] = s_sum;
        }
    }
}

// Merge of the split records of one (sequence, query head); thread = dim.
// [Day 9-2] §2 segment 3 generalised to several partial states:
// M = max_i M_i, S = sum_i S_i 2^(M_i - M), out = sum_i acc_i 2^(M_i - M) / S.
__global__ void __launch_bounds__(kHD)
decode_combine_kernel(DecodeParams p, int G) {
    const int qh = blockIdx.x, b = blockIdx.y, i = threadIdx.x;
    const int h = qh / G, g = qh % G;
    const int cap = p.max_blocks * kBS;
    const int L = max(0, min(p.ctx_lens[b], cap));
    const int split_tokens = p.split_blocks * kBS;
    const int nvalid = (L + split_tokens - 1) / split_tokens;
    const size_t rec0 = ((size_t)b * p.nkv + h) * p.nsplit;

    float m = -INFINITY;
    for (int j = 0; j < nvalid; ++j) m = fmaxf(m, p.ws_ml[((rec0 + j) * G + g) * 2]);
    float s_sum = 0.0f, a = 0.0f;
    if (m != -INFINITY) {
        for (int j = 0; j < nvalid; ++j) {
            const size_t r = (rec0 + j) * G + g;
            const float f = exp2f(p.ws_ml[r * 2] - m);
            s_sum += p.ws_ml[r * 2 + 1] * f;
            a += p.ws_acc[r * kHD + i] * f;
        }
    }
    p.out[((size_t)b * p.nqh + qh) * kHD + i] = s_sum > 0.0f ? a / s_sum : 0.0f;
}

}  // namespace

// The split size aims at enough CTAs for several waves on a 152-SM GB300
// while keeping each split long (partials stay well under 1% of KV bytes).
bool make_decode_plan(int batch, int nqh, int nkv, int max_blocks, DecodePlan *plan) {
    if (batch < 0 || nqh <= 0 || nkv <= 0 || max_blocks <= 0 || nqh % nkv) return false;
    const int G = nqh / nkv;
    const int64_t units = (int64_t)batch * nkv;
    const int64_t target_ctas = 152 * 8;
    int64_t sb = (units * max_blocks + target_ctas - 1) / target_ctas;
    sb = sb < 1 ? 1 : (sb > 16 ? 16 : sb);
    plan->group = G;
    plan->split_blocks = (int)sb;
    plan->nsplit = (int)((max_blocks + sb - 1) / sb);
    plan->records = units * plan->nsplit;
    auto align = [](size_t x) { return (x + 255) & ~(size_t)255; };
    plan->ml_offset = 0;
    plan->acc_offset = align((size_t)plan->records * G * 2 * sizeof(float));
    plan->bytes = plan->acc_offset + align((size_t)plan->records * G * kHD * sizeof(float));
    if (plan->bytes == 0) plan->bytes = 256;
    return true;
}

cudaError_t launch_decode_split(const DecodeParams &p, int group, cudaStream_t s) {
    dim3 grid(p.nsplit, p.nkv, p.batch);
    switch (group) {
        case 1: decode_split_kernel<1><<<grid, kWarps * 32, 0, s>>>(p); break;
        case 2: decode_split_kernel<2><<<grid, kWarps * 32, 0, s>>>(p); break;
        case 4: decode_split_kernel<4><<<grid, kWarps * 32, 0, s>>>(p); break;
        case 8: decode_split_kernel<8><<<grid, kWarps * 32, 0, s>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_decode_combine(const DecodeParams &p, int group, cudaStream_t s) {
    dim3 grid(p.nqh, p.batch);
    decode_combine_kernel<<<grid, kHD, 0, s>>>(p, group);
    return cudaGetLastError();
}

}  // namespace kvq8
