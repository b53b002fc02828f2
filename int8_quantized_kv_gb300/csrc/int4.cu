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
// Cache layout (per (block, kv head) tile of 256 tokens); a code byte is
// always the page's pair, byte i = code[2i] << 4 | code[2i+1]:
//   K codes uint8 [256][64]            token-major rows
//   V codes uint8 [8][64][32]          per 32-token chunk, byte column c (dims 2c,
//                                      2c+1) of the chunk's tokens, token t at
//                                      position v4_pos(t) (below)
//   params  fp32  [256][4]             (scale of dims 0-63, its zero, scale of
//                                      64-127, its zero), for K and for V
// 160 bytes per (token, kv head).
//
// Decode: one CTA per (split, kv head, sequence), 4 warps walking the split in
// 32-token chunks (each staged by bulk copies), each warp with its own
// online-softmax state.  Both contractions run on the tensor cores with the
// codes as fp16 subnormals (the tensor-core decode section below); the score
// is s = sm_scale * sum_g scale_g * (sum_{d in g} q_d c_d - zero_g *
// sum_{d in g} q_d), i.e. exactly q . dequant(k).  The warps' states are merged
// into one partial record per query head, in the record format of the q8
// decode, so the same combine kernel finishes it.
#include <cuda_fp16.h>
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

// Quantises one row (lane l holds dims 4l..4l+3): returns the lane's two code
// bytes (dims 4l, 4l+1 in the low byte, 4l+2, 4l+3 in the high byte) and
// stores the row's parameters.  A 64-value group holding a NaN or an infinity
// (outside the rule) is quantised as a group of zeros (scale 1, zero -0,
// codes 0) and KVQ8_DEV_NONFINITE is set in *status (when non-null).
__device__ __forceinline__ uint32_t int4_quant_row(float4 x, float *param_row, int lane, uint32_t *status) {
    const uint32_t bad = __ballot_sync(0xffffffffu, nonfinite(x.x) | nonfinite(x.y) | nonfinite(x.z) |
                                                        nonfinite(x.w));
    if (bad & (lane < 16 ? 0x0000ffffu : 0xffff0000u)) {   // uniform within the half warp
        x = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if ((lane & 15) == 0) flag_status(status, KVQ8_DEV_NONFINITE);
    }
    float mx = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
    float mn = fminf(fminf(x.x, x.y), fminf(x.z, x.w));
    mx = half_max(mx);
    mn = half_min(mn);
    const float s = (mx != mn) ? __fdiv_rn(__fsub_rn(mx, mn), 15.0f) : 1.0f;
    const float z = rintf(__fdiv_rn(-mn, s));
    const int c0 = int4_code(x.x, s, z), c1 = int4_code(x.y, s, z);
    const int c2 = int4_code(x.z, s, z), c3 = int4_code(x.w, s, z);
    if ((lane & 15) == 0) {
        param_row[(lane >> 4) * 2 + 0] = s;
        param_row[(lane >> 4) * 2 + 1] = z;
    }
    return (uint32_t)(((c0 << 4) | c1) | (((c2 << 4) | c3) << 8));
}

// Position of token t (0..31) of a chunk in its V byte column: the word
// 2*t4 + k of the column holds, in bytes 0..3, the tokens 16k + 2*t4 + {0, 8,
// 1, 9} -- so that in the P.V MMA (k index = token within the 16-token step)
// lane t4's one 64-bit load gives, for both k-steps, the A-fragment pairs
// {k = 2*t4, 2*t4 + 1} (bytes 0, 2) and {2*t4 + 8, 2*t4 + 9} (bytes 1, 3).
__host__ __device__ __forceinline__ int v4_pos(int t) {
    const int k = t >> 4, r = t & 15;
    return 4 * (2 * ((r & 7) >> 1) + k) + 2 * (r & 1) + (r >> 3);
}

// Stores one quantised row (the lane's two code bytes) as a K row (token-major)
// or into the V chunk layout at tile slot `slot`.
__device__ __forceinline__ void int4_store_k_row(uint32_t two, uint8_t *codes_row, int lane) {
    reinterpret_cast<uint16_t *>(codes_row)[lane] = (uint16_t)two;
}
__device__ __forceinline__ void int4_store_v_row(uint32_t two, uint8_t *v_tile, int slot, int lane) {
    uint8_t *col = v_tile + (size_t)(slot >> 5) * (kChunk4 * kRowBytes) + v4_pos(slot & 31);
    col[(size_t)(2 * lane) * kChunk4] = (uint8_t)(two & 0xff);
    col[(size_t)(2 * lane + 1) * kChunk4] = (uint8_t)(two >> 8);
}

// One warp per new (token, kv head): K row then V row.
__global__ void __launch_bounds__(kAppendWarps4 * 32)
int4_append_kernel(Int4AppendParams p) {
    // A programmatic dependent of the kernel before it, whose outputs it may
    // read: it waits for it first.  The next kernel (a decode's split, which
    // waits for this one before it reads anything) may launch at once.
    pdl_wait();
    pdl_launch_dependents();
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
    const size_t tile = (size_t)phys * p.nkv + h;
    const size_t row = tile * kBS + pos % kBS;
    const size_t src = (((size_t)b * p.n_new + i) * p.nkv + h) * kHD;
    int4_store_k_row(int4_quant_row(reinterpret_cast<const float4 *>(p.k_new + src)[lane], p.k_param + row * 4,
                                    lane, p.dev_status),
                     p.k_codes + row * kRowBytes, lane);
    int4_store_v_row(int4_quant_row(reinterpret_cast<const float4 *>(p.v_new + src)[lane], p.v_param + row * 4,
                                    lane, p.dev_status),
                     p.v_codes + tile * kBS * kRowBytes, pos % kBS, lane);
}

// ---- requantisation int8 -> INT4 of whole blocks (mixed precision by token age) ----
// [UltraQuant] §3.3 ("practical note"): the oldest time blocks are requantised
// from 8-bit to 4-bit.  Value of an int8 code: code * scale (fp32); then the
// group-64 rule above.  One CTA per (block, kv head) tile of 256 tokens; K
// rows are read chunk by chunk (undoing the slot-dependent chunk order), V
// quarters ([128 dims][64 tokens]) are transposed through shared memory.
constexpr int kReqWarps = 8;
constexpr int kVtPitch = 65;   // odd byte pitch: lane l's rows fall in distinct banks

__global__ void __launch_bounds__(kReqWarps * 32)
int4_requantize_kernel(Int4RequantParams p) {
    __shared__ uint8_t vt[kHD * kVtPitch];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y, b = blockIdx.z;
    const int from = p.blk_from[b], to = p.blk_to[b];
    if (blockIdx.x == 0 && threadIdx.x == 0 &&
        (from < 0 || to > p.max_blocks || to - from > p.max_count))
        flag_status(p.dev_status, KVQ8_DEV_BAD_POSITION);
    const int j = max(0, from) + blockIdx.x;
    if (j >= min(to, p.max_blocks)) return;
    const int phys8 = p.table8[(size_t)b * p.max_blocks + j];
    const int phys4 = p.table4[(size_t)b * p.max_blocks + j];
    if (phys8 < 0 || phys8 >= p.num_blocks8 || phys4 < 0 || phys4 >= p.num_blocks4) {
        if (threadIdx.x == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_BLOCK_ID);
        return;
    }
    const size_t tile8 = (size_t)phys8 * p.nkv + h, tile4 = (size_t)phys4 * p.nkv + h;
    // K: lane l takes dims 4l..4l+3 (logical chunk l/4, stored at chunk (l/4) ^ (t & 7))
    for (int t = warp; t < kBS; t += kReqWarps) {
        const int8_t *row = p.k_pool + (tile8 * kBS + t) * kHD;
        const uint32_t w = *reinterpret_cast<const uint32_t *>(row + 16 * ((lane >> 2) ^ (t & 7)) + 4 * (lane & 3));
        const float sc = p.k_scale[tile8 * kBS + t];
        const float4 x = make_float4(__fmul_rn((float)(int8_t)(w & 0xff), sc), __fmul_rn((float)(int8_t)((w >> 8) & 0xff), sc),
                                     __fmul_rn((float)(int8_t)((w >> 16) & 0xff), sc), __fmul_rn((float)(int8_t)(w >> 24), sc));
        int4_store_k_row(int4_quant_row(x, p.k_param + (tile4 * kBS + t) * 4, lane, p.dev_status),
                         p.k_codes + (tile4 * kBS + t) * kRowBytes, lane);
    }
    // V: one 64-token quarter at a time
    for (int qd = 0; qd < kBS / kStageTok; ++qd) {
        const uint8_t *src = reinterpret_cast<const uint8_t *>(p.v_pool) + tile8 * kHD * kBS + qd * kTileVQuarter;
        __syncthreads();
        for (int i = threadIdx.x; i < kHD * kStageTok / 16; i += kReqWarps * 32) {
            const int4 v = reinterpret_cast<const int4 *>(src)[i];
            const int r = (16 * i) / kStageTok, c0 = (16 * i) % kStageTok;
            const uint32_t ws[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
#pragma unroll
            for (int k = 0; k < 16; ++k) vt[r * kVtPitch + c0 + k] = (uint8_t)(ws[k >> 2] >> (8 * (k & 3)));
        }
        __syncthreads();
        for (int tq = warp; tq < kStageTok; tq += kReqWarps) {
            const int t = qd * kStageTok + tq;
            const float sc = p.v_scale[tile8 * kBS + t];
            float xs[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) xs[i] = __fmul_rn((float)(int8_t)vt[(4 * lane + i) * kVtPitch + tq], sc);
            int4_store_v_row(int4_quant_row(make_float4(xs[0], xs[1], xs[2], xs[3]),
                                            p.v_param + (tile4 * kBS + t) * 4, lane, p.dev_status),
                             p.v_codes + tile4 * kBS * kRowBytes, t, lane);
        }
    }
}

// ---- tensor-core decode ----
// Both contractions run as mma.sync m16n8k16 (fp16 in, fp32 accumulate).
// Codes enter as fp16 by one mask per two codes, with no conversion: the
// masked bits of a low nibble are the fp16 subnormal c * 2^-24, those of a
// high nibble, in place, 16c * 2^-24 (exact); the sums are scaled back by 2^24.
//
// Q.K as S = K Q^T: A = K codes (rows = 16 tokens, k = dims), B = the fp32
// query split into fp16 high + low parts (columns = heads).  The query values
// facing high nibbles are divided by 16, so each code meets its own q:
//   s = sm * 2^-k * sum_g scale_g * (2^24 D'_g - zero_g Q_g),
//   D'_g = sum_{d in g} a_d y_d,  Q_g = sum_{d in g} q_d,
// a = the fed code value, y = the fed query value (q or q/16, as high + low
// fp16 parts), q = the query times a power of two 2^k that puts its largest
// element at 2^13..2^14 (fp16 keeps full precision for q/16).  The score
// fragment (row = token, column = head) reaches P.V through shared memory: P'
// is stored as fp16 tiles of 32 tokens x 8 columns in the chunk's K area
// (free once K has been read) and loaded back transposed (ldmatrix .trans)
// into the B fragments.
//
// P.V as out^T = V^T P: A = V codes (rows = dims, k = tokens), B = P'_g = w *
// vscale_g(t) * 2^-e per dim group, split into fp16 high + low; the high
// nibble of a byte enters as 16c, which the epilogue divides by 16; the zero
// point enters as a correction per (head, group),
//   out[d][h] = 2^24 sum_t P'_g a_{t,d} - Z[h][g],  Z[h][g] = sum_t P'_g zero_g(t),
// rescaled with the accumulator.  Row r of m-tile mt is dim 2*B + (r >= 8)
// with byte column B = 8*mt + r%8 of the chunk's dim-major V layout, so one
// 64-bit load per lane and m-tile feeds both k-steps (v4_pos), with no byte
// permutes, and the loads of a half warp fall in distinct banks.
//
// k-order of Q.K (k-step ks: group ks/4, sub = ks%4; lane t4 supplies the
// nibbles of the word at byte 32*(ks/4) + 8*t4 + 4*(sub/2)): k = 2*t4 + e ->
// the high nibble of byte (sub%2) + 2e, k = 2*t4 + 8 + e -> its low nibble.
// The fp16 pair {n0 * 2^-24, n2 * 2^-24} of the low nibbles of bytes 0 and 2
// of w (mask 0x000F000F), or {16 n0' * 2^-24, 16 n2' * 2^-24} of their high
// nibbles (mask 0x00F000F0): the masked bits are fp16 subnormals, exact.
__device__ __forceinline__ uint32_t nib_pair(uint32_t w, uint32_t mask) { return w & mask; }
constexpr float kNibUnit = 0x1p24f;   // 1 / the value of one code step in nib_pair
constexpr uint32_t kLoNib = 0x000F000Fu, kHiNib = 0x00F000F0u;

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// dim of k index kk (0..15) of Q.K k-step ks
__device__ __forceinline__ int qk_dim(int ks, int kk) {
    const int gr = ks >> 2, sub = ks & 3, t4 = (kk & 7) >> 1, e = kk & 1, lo = kk >> 3;
    const int byte = 32 * gr + 8 * t4 + 4 * (sub >> 1) + (sub & 1) + 2 * e;
    return 2 * byte + lo;
}

// Per-warp staging of one 32-token chunk: its K codes (2 KiB), V codes (2 KiB)
// and K and V parameter rows (512 B each) are contiguous in the cache (a chunk
// starts at a multiple of 32 slots), so one lane brings each in with a 1-D
// bulk copy, completing on the buffer's mbarrier; two buffers per warp.  The
// staged K rows keep the cache's 64-byte pitch; their fragment loads meet
// 2-way bank conflicts, which cost nothing measurable (a cache layout that
// removed them, with the rows' 32-byte pieces permuted, ran at the same speed).
constexpr int kStageKOff = 0;
constexpr int kStageVOff = kChunk4 * kRowBytes;                   // 2048
constexpr int kStageKpOff = kStageVOff + kChunk4 * kRowBytes;     // 4096
constexpr int kStageVpOff = kStageKpOff + kChunk4 * 16;           // 4608
constexpr int kStageBytes4 = kStageVpOff + kChunk4 * 16;          // 5120
constexpr int kBufs4 = 2;
constexpr uint64_t kWait4Ns = 2000000000ull;                      // bound of every copy wait

template <int G>
struct Int4Smem {
    float qrows[G * kHD];            // the unit's query rows
    uint4 qa[8][32];                 // per k-step and lane: a0 high, a2 high, a0 low, a2 low
    float qq[8][2];                  // Q_g per head
    float qmax[kWarps4];
    unsigned long long bar[kWarps4][kBufs4];   // per warp and buffer: copies complete
    union {
        unsigned char stage[kWarps4][kBufs4][kStageBytes4];
        struct {
            float acc[kWarps4][G][kHD];
            float ml[kWarps4][G][2];
        } red;
    } u;
};

// Fills `buf` (its mbarrier `bar`) with chunk `cidx` of this warp's split:
// lane 0 issues the four bulk copies, or, when the chunk does not exist or its
// block id is invalid, completes the barrier's phase with a plain arrival.
// The block id of logical block hint_lb is hint_phys (loaded earlier; -1: no
// hint).
// Every call completes exactly one phase of `bar`.  Returns the block id (-1
// for no data).  The buffer's earlier contents were read and written through
// the generic proxy; the proxy fence orders those accesses (of every lane: the
// caller synchronises the warp first) before the copies' writes.
__device__ __forceinline__ int int4_fetch_chunk(const Int4DecodeParams &p, int b, int h, int tok_begin,
                                                int nchunks, int cidx, unsigned char *buf, uint32_t bar,
                                                uint64_t pol, int lane, int hint_lb = -1, int hint_phys = -1) {
    int phys = -1;
    if (cidx < nchunks) {
        const int t0 = tok_begin + cidx * kChunk4;
        phys = t0 / kBS == hint_lb ? hint_phys : p.block_table[(size_t)b * p.max_blocks + t0 / kBS];
        if (phys < 0 || phys >= p.num_blocks) {
            if (lane == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_BLOCK_ID);
            phys = -1;
        } else if (lane == 0) {
            const size_t row0 = ((size_t)phys * p.nkv + h) * kBS + t0 % kBS;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive_expect_tx(bar, kStageBytes4);
            bulk_copy_g2s(smem_addr(buf + kStageKOff), p.k_codes + row0 * kRowBytes, kChunk4 * kRowBytes, bar, pol);
            bulk_copy_g2s(smem_addr(buf + kStageVOff), p.v_codes + row0 * kRowBytes, kChunk4 * kRowBytes, bar, pol);
            bulk_copy_g2s(smem_addr(buf + kStageKpOff), p.k_param + row0 * 4, kChunk4 * 16, bar, pol);
            bulk_copy_g2s(smem_addr(buf + kStageVpOff), p.v_param + row0 * 4, kChunk4 * 16, bar, pol);
        }
    }
    if (phys < 0 && lane == 0) mbar_arrive(bar);
    return phys;
}

// A decode step's new token of unit (b, h), position pos = ctx_lens[b] - 1,
// which is row t of the chunk staged at st: quantised by the warp (the group-64
// rule of int4_append_kernel), written over the row the copy brought in (K
// row, the V chunk's columns at v4_pos(t), both parameter rows) and into the
// cache.  Only this warp reads that position in this launch.
__device__ __noinline__ void int4_append_new_token(const Int4DecodeParams &p, int b, int h, int pos, int t,
                                                   int lane, unsigned char *st) {
    const int phys = p.block_table[(size_t)b * p.max_blocks + pos / kBS];   // valid: the chunk was staged
    const size_t tile = (size_t)phys * p.nkv + h;
    const size_t row = tile * kBS + pos % kBS;
    const size_t src = ((size_t)b * p.nkv + h) * kHD;
    float *kpar = reinterpret_cast<float *>(st + kStageKpOff) + 4 * t;
    float *vpar = reinterpret_cast<float *>(st + kStageVpOff) + 4 * t;
    const uint32_t kt = int4_quant_row(reinterpret_cast<const float4 *>(p.k_new + src)[lane], kpar, lane,
                                       p.dev_status);
    const uint32_t vt = int4_quant_row(reinterpret_cast<const float4 *>(p.v_new + src)[lane], vpar, lane,
                                       p.dev_status);
    // the staged chunk
    int4_store_k_row(kt, st + kStageKOff + t * kRowBytes, lane);
    st[kStageVOff + (2 * lane) * kChunk4 + v4_pos(t)] = (uint8_t)(vt & 0xff);
    st[kStageVOff + (2 * lane + 1) * kChunk4 + v4_pos(t)] = (uint8_t)(vt >> 8);
    // the cache (the pools of a decode step are the caller's writable buffers)
    int4_store_k_row(kt, const_cast<uint8_t *>(p.k_codes) + row * kRowBytes, lane);
    int4_store_v_row(vt, const_cast<uint8_t *>(p.v_codes) + tile * kBS * kRowBytes, pos % kBS, lane);
    __syncwarp();   // the parameter rows written by lanes 0 and 16
    if (lane < 4) {
        const_cast<float *>(p.k_param)[row * 4 + lane] = kpar[lane];
        const_cast<float *>(p.v_param)[row * 4 + lane] = vpar[lane];
    }
    __syncwarp();   // the patched chunk is read by every lane below
}

template <int G, bool kStep>
__global__ void __launch_bounds__(kWarps4 * 32, 3)
int4_decode_split_kernel(Int4DecodeParams p) {
    // kPack (G <= 4): the 8 MMA columns carry both fp16 parts (high, low) of
    // the operand facing the heads, so one MMA does both halves.  kPackH
    // (G = 4): column 2j + e is part e of head j, so lane (g, t4) holds both
    // parts of head t4 (scores of tokens 16*mt + g + 8*r, accumulator columns),
    // added in the lane.  kPack2 (G <= 2): columns 0-1 high parts, 2-3 low
    // parts, 4-7 zero; one shuffle joins the halves (lanes t4 = 0, 1 keep rows g, g + 8) and a
    // second moves the second m-tile's scores to lanes t4 = 2, 3, so that lane
    // (g, t4) owns token 16*(t4/2) + g + 8*(t4%2) and both heads: no lane
    // works on padding heads.  Otherwise (G = 8) the columns are the 8 heads
    // and each product takes two MMAs.
    constexpr bool kPack = G <= 4;
    constexpr bool kPack2 = G <= 2;
    constexpr bool kPackH = kPack && !kPack2;
    constexpr int kHL = kPackH ? 1 : 2;   // heads per lane
    pdl_wait();
    // In a mixed-precision decode the next kernel is the int8 split over the
    // recent tokens, which reads nothing this kernel writes: it may start now
    // and take the SMs this grid leaves (it waits for this grid before it
    // completes, so the merge after it sees both splits' records).
    if (p.n4_blocks) pdl_launch_dependents();
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int cap = p.max_blocks * kBS;
    // the unit's query rows, loaded beside the context length (no load of
    // the prologue waits for another but the block id after the length)
    constexpr int kQV = (G * 32 + kWarps4 * 32 - 1) / (kWarps4 * 32);   // float4 per thread
    const float4 *qsrc = reinterpret_cast<const float4 *>(p.q + ((size_t)b * p.nqh + (size_t)h * G) * kHD);
    float4 qv[kQV];
#pragma unroll
    for (int r = 0; r < kQV; ++r) {
        const int i = threadIdx.x + r * kWarps4 * 32;
        qv[r] = i < G * 32 ? qsrc[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // the block ids of this warp's first chunks, loaded beside the length too,
    // for a unit that fills the table (the usual case outside a mixed-precision
    // decode); used only when the length confirms where the split starts
    const int st_full = int4_split_tokens(cap, p.nsplit);
    int hint_lb[kBufs4], hint_phys[kBufs4];
#pragma unroll
    for (int i = 0; i < kBufs4; ++i) {
        const int lb = (split * st_full + kChunk4 * (warp + kWarps4 * i)) / kBS;
        hint_lb[i] = (!p.n4_blocks && lb < p.max_blocks) ? lb : -1;
        hint_phys[i] = hint_lb[i] >= 0 ? p.block_table[(size_t)b * p.max_blocks + lb] : -1;
    }
    int L = p.ctx_lens[b];
    // a decode step appends its new token at position ctx_lens[b] - 1 (none
    // for an empty context or one beyond the table)
    const int app_pos = (kStep && L >= 1 && L <= cap) ? L - 1 : -1;
    if (L < 0 || L > cap) {
        if (threadIdx.x == 0 && split == 0 && h == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_CTX_LEN);
        L = max(0, min(L, cap));
    }
    if (p.n4_blocks) L = min(L, max(0, min(p.n4_blocks[b], p.max_blocks)) * kBS);   // the 4-bit part only
    const size_t u = (size_t)b * p.nkv + h;
    // this unit's nsplit splits share its L tokens evenly (whole chunks), so
    // that a unit shorter than the table (a short context, or the 4-bit part
    // of a mixed-precision sequence) still keeps every CTA of the grid busy
    const int st = int4_split_tokens(L, p.nsplit);
    static_assert(kChunk4 == 32, "int4_split_tokens cuts units into 32-token chunks");
    if (split == 0 && threadIdx.x == 0) {
        // records of unit u are u*nsplit + j; the combine reads first + u + j
        p.ws_meta[u] = make_int2((int)(u * (p.nsplit - 1)), int4_split_count(L, p.nsplit));
    }
    const int tok_begin = split * st;
    if (tok_begin >= L) return;
    const int tok_end = min(L, tok_begin + st);

    extern __shared__ __align__(16) unsigned char int4_smem_raw[];
    Int4Smem<G> &sm = *reinterpret_cast<Int4Smem<G> *>(int4_smem_raw);
    // this warp's chunks: cidx = warp, warp + 4, ...; two in flight.  Bit i of
    // `valid`: buffer i holds a chunk; of `fill_par`: parity of the phase of
    // buffer i's latest fill; of `pending`: that phase is not waited for yet
    const int nchunks = (tok_end - tok_begin + kChunk4 - 1) / kChunk4;
    const uint64_t pol = l2_evict_first_policy();
    const uint32_t bar0 = smem_addr(&sm.bar[warp][0]);
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < kBufs4; ++i) mbar_init(bar0 + 8 * i, 1);
        fence_mbar_init();
    }
    __syncwarp();
    unsigned valid = 0, fill_par = 0, pending = (1u << kBufs4) - 1;
    const bool hinted = st == st_full;   // the split starts where the hints assumed
#pragma unroll
    for (int i = 0; i < kBufs4; ++i)
        valid |= (unsigned)(int4_fetch_chunk(p, b, h, tok_begin, nchunks, warp + kWarps4 * i, sm.u.stage[warp][i],
                                             bar0 + 8 * i, pol, lane, hinted ? hint_lb[i] : -1,
                                             hint_phys[i]) >= 0) << i;
    bool aborted = false;

    const float *qrow = sm.qrows;
    // power of two 2^k with max |q| * 2^k in [2^13, 2^14)
    {
        float m = 0.0f;
#pragma unroll
        for (int r = 0; r < kQV; ++r) {
            const int i = threadIdx.x + r * kWarps4 * 32;
            if (i < G * 32) reinterpret_cast<float4 *>(sm.qrows)[i] = qv[r];
            m = fmaxf(m, fmaxf(fmaxf(fabsf(qv[r].x), fabsf(qv[r].y)), fmaxf(fabsf(qv[r].z), fabsf(qv[r].w))));
        }
        m = warp_max(m);
        if (lane == 0) sm.qmax[warp] = m;
    }
    __syncthreads();
    float qmax = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps4; ++w) qmax = fmaxf(qmax, sm.qmax[w]);
    // 2^qk with qk = 13 - ilogb(max |q|), clamped to [-120, 120], built from
    // the exponent bits (a subnormal maximum reads as 2^-127: clamped alike)
    const int qexp = (qmax > 0.0f && isfinite(qmax)) ? 13 - ((int)((__float_as_uint(qmax) >> 23) & 0xff) - 127) : 0;
    const int qk = max(-120, min(120, qexp));
    const float qscale = __int_as_float((127 + qk) << 23);
    // B fragments of Q in the Q.K k-order (column gg of lane (gg, tt); the
    // values facing high nibbles, k = 2*tt + e, carry q / 16).  kPack: kept in
    // registers, column gg = head gg % 4, high part for gg < 4, low part else;
    // otherwise staged in shared memory as high and low parts of head gg.
    uint32_t qb[8][2];
    if constexpr (kPack) {
        // kPack2: column gg = head gg % 2 (gg < 4; high part for gg < 2), zero
        // for gg >= 4; kPackH: head gg / 2, high part for even gg
        const int hq = kPack2 ? (g < 4 ? (g & 1) : G) : (g >> 1);
        const bool low = kPack2 ? (g & 2) != 0 : (g & 1) != 0;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            float x[4] = {0.f, 0.f, 0.f, 0.f};
            if (hq < G) {
                const float *qg = qrow + (size_t)hq * kHD;
                x[0] = qg[qk_dim(ks, 2 * t4)] * qscale * 0.0625f;
                x[1] = qg[qk_dim(ks, 2 * t4 + 1)] * qscale * 0.0625f;
                x[2] = qg[qk_dim(ks, 2 * t4 + 8)] * qscale;
                x[3] = qg[qk_dim(ks, 2 * t4 + 9)] * qscale;
            }
            float y[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float hi = __half2float(__float2half_rn(x[e]));
                y[e] = low ? x[e] - hi : hi;
            }
            qb[ks][0] = pack_half2(y[0], y[1]);
            qb[ks][1] = pack_half2(y[2], y[3]);
        }
    } else {
        for (int i = threadIdx.x; i < 8 * 32; i += kWarps4 * 32) {
            const int ks = i >> 5, ln = i & 31, gg = ln >> 2, tt = ln & 3;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (gg < G) {
                const float *qg = qrow + (size_t)gg * kHD;
                const float x0 = qg[qk_dim(ks, 2 * tt)] * qscale * 0.0625f;
                const float x1 = qg[qk_dim(ks, 2 * tt + 1)] * qscale * 0.0625f;
                const float x8 = qg[qk_dim(ks, 2 * tt + 8)] * qscale, x9 = qg[qk_dim(ks, 2 * tt + 9)] * qscale;
                const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
                const __half h8 = __float2half_rn(x8), h9 = __float2half_rn(x9);
                v.x = pack_half2(__half2float(h0), __half2float(h1));
                v.y = pack_half2(__half2float(h8), __half2float(h9));
                v.z = pack_half2(x0 - __half2float(h0), x1 - __half2float(h1));
                v.w = pack_half2(x8 - __half2float(h8), x9 - __half2float(h9));
            }
            sm.qa[ks][ln] = v;
        }
    }
    {
        // Q_g: 8 threads per (head, group), 8 dims each, summing the query as
        // the MMAs see it (even dims face high nibbles and are fed as q / 16,
        // as high + low fp16 parts)
        const int gg = threadIdx.x >> 4, gr = (threadIdx.x >> 3) & 1, part = threadIdx.x & 7;
        float qs = 0.0f;
        if (gg < G) {
#pragma unroll
            for (int d = 0; d < 8; ++d) {
                const int dim = 64 * gr + 8 * part + d;
                const float f = (dim & 1) ? 1.0f : 0.0625f;
                const float x = qrow[(size_t)gg * kHD + dim] * qscale * f;
                const float hf = __half2float(__float2half_rn(x));
                const float y = hf + __half2float(__float2half_rn(x - hf));
                qs += y / f;
            }
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) qs += __shfl_xor_sync(0xffffffffu, qs, o);
        if (part == 0) sm.qq[gg][gr] = qs;
    }
    __syncthreads();
    // this lane's heads (score and accumulator columns): 2*(t4 % 2) + j when
    // packed, 2*t4 + j otherwise
    const int hbase = kPack2 ? 0 : (kPackH ? t4 : 2 * t4);
    float qq[2][2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int gr = 0; gr < 2; ++gr) qq[j][gr] = sm.qq[hbase + j][gr];
    const float score_scale = p.sm_scale_log2 * __int_as_float((127 - qk) << 23);   // / qscale, exactly

    // scores per lane: kPack2 1 token x 2 heads, kPackH 4 tokens (rows g, g + 8
    // of both m-tiles) x 1 head, else 4 tokens x 2 heads
    constexpr int kR = kPack2 ? 1 : 2;
    constexpr int kM = kPack2 ? 1 : 2;   // score m-slots per lane
    const int tok2 = 16 * (t4 >> 1) + g + 8 * (t4 & 1);   // kPack2: this lane's token
    float M[2] = {-INFINITY, -INFINITY}, Sl[2] = {0.0f, 0.0f}, Zl[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};
    float acc[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mt][i] = 0.0f;
    int e_cur = 1000;   // acc and Zl hold values in units of 2^e_cur

    for (int it = 0, cidx = warp; cidx < nchunks; ++it, cidx += kWarps4) {
        const int bi = it % kBufs4;
        if (!mbar_wait_bounded(bar0 + 8 * bi, (fill_par >> bi) & 1u, kWait4Ns)) {
            if (lane == 0) flag_status(p.dev_status, KVQ8_DEV_TIMEOUT);
            aborted = true;
            break;
        }
        pending &= ~(1u << bi);
        __syncwarp();
        const unsigned char *st = sm.u.stage[warp][bi];
        if ((valid >> bi) & 1u) {
        const int t0 = tok_begin + cidx * kChunk4;
        const int ntok = min(kChunk4, tok_end - t0);
        if constexpr (kStep) {
            if (app_pos >= t0 && app_pos < t0 + ntok)
                int4_append_new_token(p, b, h, app_pos, app_pos - t0, lane, const_cast<unsigned char *>(st));
        }
        const float4 *kps = reinterpret_cast<const float4 *>(st + kStageKpOff);
        const float4 *vps = reinterpret_cast<const float4 *>(st + kStageVpOff);
        // K rows, V words and parameters are read from the staging buffer just
        // before their use (short register lifetimes)
        const bool partial = ntok < kChunk4;   // only the split's last chunk

        // ---- scores: S = K Q^T, tokens 16*mt + g + 8*r (rows) ----
        float sc[kM][kR][2];
        float mloc[2] = {-INFINITY, -INFINITY};
        float dtm[2][2][2];   // kPack2: [m-tile][group][head] sums of this lane's row
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            // K: tokens 16*mt + g + 8*r, bytes 32*gr + 8*t4 .. +7
            uint2 kw[2][2];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int gr = 0; gr < 2; ++gr) {
                    const int t = 16 * mt + g + 8 * r;
                    kw[r][gr] = *reinterpret_cast<const uint2 *>(st + kStageKOff + t * kRowBytes + 32 * gr + 8 * t4);
                }
            float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};   // per group
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int gr = ks >> 2, sub = ks & 3;
                uint32_t a[4];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint32_t w0 = (sub >> 1) ? kw[r][gr].y : kw[r][gr].x;
                    const uint32_t w = (sub & 1) ? (w0 >> 8) : w0;
                    a[r] = nib_pair(w, kHiNib);       // rows g / g+8, k = 2*t4 + e
                    a[2 + r] = nib_pair(w, kLoNib);   // rows g / g+8, k = 2*t4 + 8 + e
                }
                if constexpr (kPack) {
                    mma_f16_16816(d[gr], a[0], a[1], a[2], a[3], qb[ks][0], qb[ks][1]);
                } else {
                    const uint4 qa = sm.qa[ks][lane];
                    mma_f16_16816(d[gr], a[0], a[1], a[2], a[3], qa.x, qa.y);
                    mma_f16_16816(d[gr], a[0], a[1], a[2], a[3], qa.z, qa.w);
                }
            }
            if constexpr (kPack2) {
                // lane t4 = 0 holds the high parts of rows g and g + 8, lane 1 the
                // low parts: each keeps one row (t4 = 0: g) and receives the other
                // part; lanes t4 = 2, 3 hold the zero columns
                const bool lo_lane = (t4 & 1) != 0;
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int gr = 0; gr < 2; ++gr) {
                        const float send = lo_lane ? d[gr][j] : d[gr][2 + j];
                        const float keep = lo_lane ? d[gr][2 + j] : d[gr][j];
                        dtm[mt][gr][j] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
                    }
            } else if constexpr (kPackH) {
                // columns 2*t4, 2*t4 + 1: the high and low parts of head t4, rows
                // g and g + 8
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float4 k4 = kps[16 * mt + g + 8 * r];
                    const float dt0 = d[0][2 * r] + d[0][2 * r + 1];
                    const float dt1 = d[1][2 * r] + d[1][2 * r + 1];
                    const float x = k4.x * fmaf(dt0, kNibUnit, -k4.y * qq[0][0]) +
                                    k4.z * fmaf(dt1, kNibUnit, -k4.w * qq[0][1]);
                    sc[mt][r][0] = x * score_scale;
                }
            } else {
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    const float4 k4 = kps[16 * mt + g + 8 * r];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float x = k4.x * fmaf(d[0][2 * r + j], kNibUnit, -k4.y * qq[j][0]) +
                                        k4.z * fmaf(d[1][2 * r + j], kNibUnit, -k4.w * qq[j][1]);
                        sc[mt][r][j] = x * score_scale;
                    }
                }
            }
        }
        if constexpr (kPack2) {
            // the second m-tile's rows go to lanes t4 = 2, 3
            const float4 k4 = kps[tok2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float dt[2];
#pragma unroll
                for (int gr = 0; gr < 2; ++gr) {
                    const float m1 = __shfl_xor_sync(0xffffffffu, dtm[1][gr][j], 2);
                    dt[gr] = t4 < 2 ? dtm[0][gr][j] : m1;
                }
                const float x = k4.x * fmaf(dt[0], kNibUnit, -k4.y * qq[j][0]) +
                                k4.z * fmaf(dt[1], kNibUnit, -k4.w * qq[j][1]);
                sc[0][0][j] = x * score_scale;
            }
        }
        // token of score (mt, r) of this lane
        auto tok_of = [&](int mt, int r) { return kPack2 ? tok2 : 16 * mt + g + 8 * r; };
        if (partial) {
#pragma unroll
            for (int mt = 0; mt < kM; ++mt)
#pragma unroll
                for (int r = 0; r < kR; ++r)
                    if (tok_of(mt, r) >= ntok) {
#pragma unroll
                        for (int j = 0; j < kHL; ++j) sc[mt][r][j] = -INFINITY;
                    }
        }
        // this lane's score tokens' V parameters (zero past the end: stale slots)
        float4 vp[kM][kR];
#pragma unroll
        for (int mt = 0; mt < kM; ++mt)
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                vp[mt][r] = vps[tok_of(mt, r)];
                if (partial && tok_of(mt, r) >= ntok) vp[mt][r] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        // this lane's own maxima; the warp reduces them only when some lane's
        // score passes its head's running maximum by more than 2^8 (below)
#pragma unroll
        for (int j = 0; j < kHL; ++j)
#pragma unroll
            for (int mt = 0; mt < kM; ++mt)
#pragma unroll
                for (int r = 0; r < kR; ++r) mloc[j] = fmaxf(mloc[j], sc[mt][r][j]);

        // power-of-two unit of this chunk's P': 2^e > max V scale (see the q8 decode)
        float vsmax = 0.0f;
#pragma unroll
        for (int mt = 0; mt < kM; ++mt)
#pragma unroll
            for (int r = 0; r < kR; ++r) vsmax = fmaxf(vsmax, fmaxf(vp[mt][r].x, vp[mt][r].z));
        const int e_need = __reduce_max_sync(0xffffffffu, ((__float_as_int(vsmax) >> 23) & 0xff) - 126);
        int e_new = e_cur;
        if (e_need > e_cur || e_need < e_cur - 12) e_new = max(-120, min(120, e_need));
        const float inv = __int_as_float((127 - e_new) << 23);

        // online softmax per head (the lanes of a head agree), raised lazily:
        // some lane's score of a head is above M + 8 exactly when the head's
        // maximum over the chunk is, so the lanes' own maxima decide whether
        // to raise, and the maxima are reduced over the lanes sharing the head
        // (all g, and all lanes when kPack2) only then
        const bool grow = mloc[0] > M[0] + 8.0f || (kHL > 1 && mloc[1] > M[1] + 8.0f);
        float alpha[2] = {1.0f, 1.0f};
        bool rescale = e_new != e_cur;
        if (__any_sync(0xffffffffu, grow)) {
            rescale = true;
#pragma unroll
            for (int j = 0; j < kHL; ++j) {
                if constexpr (kPack2) mloc[j] = fmaxf(mloc[j], __shfl_xor_sync(0xffffffffu, mloc[j], 1));
                if constexpr (kPack2) mloc[j] = fmaxf(mloc[j], __shfl_xor_sync(0xffffffffu, mloc[j], 2));
                mloc[j] = fmaxf(mloc[j], __shfl_xor_sync(0xffffffffu, mloc[j], 4));
                mloc[j] = fmaxf(mloc[j], __shfl_xor_sync(0xffffffffu, mloc[j], 8));
                mloc[j] = fmaxf(mloc[j], __shfl_xor_sync(0xffffffffu, mloc[j], 16));
                const float m_new = fmaxf(M[j], mloc[j]);
                alpha[j] = exp2f(M[j] - m_new);   // 0 while M is -inf
                M[j] = m_new;
            }
        }
        const float two = __int_as_float((127 + max(-126, min(127, e_cur - e_new))) << 23);
        // P'_g = w * vscale_g * 2^-e, high and low fp16 parts, into the freed K
        // area for the transposing loads: kPackH [group][32 tokens][(high, low)
        // of heads 0-3] (kPack2: words 0, 1 = high and low parts of heads 0-1;
        // words 2, 3 unwritten, their B columns zeroed after the load), else
        // [group][part][32 tokens][8 heads]
        uint32_t *ptile = reinterpret_cast<uint32_t *>(const_cast<unsigned char *>(st) + kStageKOff);
        __syncwarp();   // every lane is done reading the K rows
        float wsum[2] = {0.f, 0.f}, zs[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
        for (int mt = 0; mt < kM; ++mt)
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                const int t = tok_of(mt, r);
                float pg[2][2];   // [group][head j]
                // the token's V scales in units of 2^e (exact: inv is a power of two)
                const float vx = vp[mt][r].x * inv, vz = vp[mt][r].z * inv;
#pragma unroll
                for (int j = 0; j < kHL; ++j) {
                    const float w = ex2_approx(sc[mt][r][j] - M[j]);   // 0 for invalid tokens (-inf)
                    wsum[j] += w;
                    pg[0][j] = w * vx;
                    pg[1][j] = w * vz;
                    zs[j][0] = fmaf(pg[0][j], vp[mt][r].y, zs[j][0]);
                    zs[j][1] = fmaf(pg[1][j], vp[mt][r].w, zs[j][1]);
                }
#pragma unroll
                for (int gr = 0; gr < 2; ++gr) {
                    if constexpr (kPackH) {
                        // word 4t + t4: the high part (low half) and the low part of
                        // this lane's head; 32 distinct banks per store
                        const float hf = __half2float(__float2half_rn(pg[gr][0]));
                        ptile[(gr * kChunk4 + t) * 4 + t4] = pack_half2(hf, pg[gr][0] - hf);
                        continue;
                    }
                    const __half2 hh = __floats2half2_rn(pg[gr][0], pg[gr][1]);
                    const float2 hf = __half22float2(hh);
                    const uint32_t hi = *reinterpret_cast<const uint32_t *>(&hh);
                    const uint32_t lo = pack_half2(pg[gr][0] - hf.x, pg[gr][1] - hf.y);
                    if constexpr (kPack2) {
                        // lanes t4 = 1, 3 store in the other order: two banks per g
                        const int w0 = t4 & 1;
                        ptile[(gr * kChunk4 + t) * 4 + w0] = w0 ? lo : hi;
                        ptile[(gr * kChunk4 + t) * 4 + (w0 ^ 1)] = w0 ? hi : lo;
                    } else {
                        ptile[((gr * 2 + 0) * kChunk4 + t) * 4 + t4] = hi;
                        ptile[((gr * 2 + 1) * kChunk4 + t) * 4 + t4] = lo;
                    }
                }
            }
#pragma unroll
        for (int j = 0; j < kHL; ++j) {
            Sl[j] = fmaf(Sl[j], alpha[j], wsum[j]);
            Zl[j][0] = fmaf(Zl[j][0], alpha[j] * two, zs[j][0]);
            Zl[j][1] = fmaf(Zl[j][1], alpha[j] * two, zs[j][1]);
        }
        if (rescale) {  // warp-uniform; accumulator columns are this lane's heads
            const float f0 = alpha[0] * two, f1 = (kPackH ? alpha[0] : alpha[1]) * two;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                acc[mt][0] *= f0; acc[mt][1] *= f1;
                acc[mt][2] *= f0; acc[mt][3] *= f1;
            }
        }
        e_cur = e_new;
        __syncwarp();
        // B fragments of P.V: matrix i of an x4 transposing load = tokens 8i..8i+7,
        // so lane (g, t4) receives {P[8i + 2*t4][g], P[8i + 2*t4 + 1][g]}
        constexpr int kParts = kPack ? 1 : 2;
        uint32_t bf[2][kParts][2][2];   // [group][part][k-step][b0, b1]
#pragma unroll
        for (int gr = 0; gr < 2; ++gr)
#pragma unroll
            for (int hl = 0; hl < kParts; ++hl) {
                const uint32_t addr = (uint32_t)__cvta_generic_to_shared(ptile + ((gr * kParts + hl) * kChunk4 + lane) * 4);
                uint32_t r0, r1, r2, r3;
                asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                             : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                             : "r"(addr));
                bf[gr][hl][0][0] = r0; bf[gr][hl][0][1] = r1; bf[gr][hl][1][0] = r2; bf[gr][hl][1][1] = r3;
                if (kPack2 && g >= 4) {   // columns 4-7: zero (the tile's words 2, 3 are stale)
                    bf[gr][hl][0][0] = 0u; bf[gr][hl][0][1] = 0u; bf[gr][hl][1][0] = 0u; bf[gr][hl][1][1] = 0u;
                }
            }

        // ---- P.V: out^T += V^T P'_g ----
        // m-tile mt: rows g, g + 8 = dims 2c, 2c + 1 of byte column c = 8*mt + g;
        // one 64-bit load gives the column's words 2*t4 (k-step 0) and 2*t4 + 1
        // (k-step 1), each holding the A fragment of one MMA: high nibbles of
        // bytes 0, 2 (rows g, k = 2*t4, 2*t4 + 1), low nibbles (rows g + 8), and
        // the same of bytes 1, 3 (k = 2*t4 + 8, 2*t4 + 9)
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int gr = mt >> 2;
            const uint2 vw = *reinterpret_cast<const uint2 *>(st + kStageVOff + (8 * mt + g) * kChunk4 + 8 * t4);
#pragma unroll
            for (int ks2 = 0; ks2 < 2; ++ks2) {
                const uint32_t w = ks2 ? vw.y : vw.x, w8 = w >> 8;
                const uint32_t a0 = nib_pair(w, kHiNib), a1 = nib_pair(w, kLoNib);
                const uint32_t a2 = nib_pair(w8, kHiNib), a3 = nib_pair(w8, kLoNib);
#pragma unroll
                for (int hl = 0; hl < kParts; ++hl)
                    mma_f16_16816(acc[mt], a0, a1, a2, a3, bf[gr][hl][ks2][0], bf[gr][hl][ks2][1]);
            }
        }
        }
        __syncwarp();
        const bool ok = int4_fetch_chunk(p, b, h, tok_begin, nchunks, cidx + kWarps4 * kBufs4,
                                         sm.u.stage[warp][bi], bar0 + 8 * bi, pol, lane) >= 0;
        valid = (valid & ~(1u << bi)) | ((unsigned)ok << bi);
        fill_par ^= 1u << bi;
        pending |= 1u << bi;
    }
    if (aborted) {
        // no copy of this warp may still be in flight when the CTA exits
#pragma unroll
        for (int i = 0; i < kBufs4; ++i)
            if ((pending >> i) & 1u) mbar_wait_bounded(bar0 + 8 * i, (fill_par >> i) & 1u, kWait4Ns);
    }

    // ---- this warp's state: the lanes of this lane's heads ----
#pragma unroll
    for (int j = 0; j < kHL; ++j) {
#pragma unroll
        for (int o = kPack2 ? 1 : 4; o < 32; o <<= 1) {
            Sl[j] += __shfl_xor_sync(0xffffffffu, Sl[j], o);
            Zl[j][0] += __shfl_xor_sync(0xffffffffu, Zl[j][0], o);
            Zl[j][1] += __shfl_xor_sync(0xffffffffu, Zl[j][1], o);
        }
    }
    if constexpr (kPack2) {
        // add the low parts' columns (lane t4 ^ 1) into the high parts'
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[mt][i] += __shfl_xor_sync(0xffffffffu, acc[mt][i], 1);
    } else if constexpr (kPackH) {
        // the low part's column (2*t4 + 1) into the high part's (2*t4), in the lane
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            acc[mt][0] += acc[mt][1];
            acc[mt][2] += acc[mt][3];
        }
    }
    const float unit_scale = __int_as_float((127 + max(-126, min(127, e_cur))) << 23);
    __syncthreads();   // every warp is done with its staging buffers
    const bool writer = kPack2 ? t4 == 0 : true;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int gr = mt >> 2;
        const int dim = 2 * (8 * mt + g);   // row g: even dim (its high nibble), row g + 8: the next
        const int h0 = hbase, h1 = hbase + 1;
        // rows g carry 16 c (high nibbles: even dims), in code steps of 2^-24
        if (writer && h0 < G) {
            sm.u.red.acc[warp][h0][dim] = fmaf(acc[mt][0], kNibUnit * 0.0625f, -Zl[0][gr]) * unit_scale;
            sm.u.red.acc[warp][h0][dim + 1] = fmaf(acc[mt][2], kNibUnit, -Zl[0][gr]) * unit_scale;
        }
        if (writer && kHL > 1 && h1 < G) {
            sm.u.red.acc[warp][h1][dim] = fmaf(acc[mt][1], kNibUnit * 0.0625f, -Zl[1][gr]) * unit_scale;
            sm.u.red.acc[warp][h1][dim + 1] = fmaf(acc[mt][3], kNibUnit, -Zl[1][gr]) * unit_scale;
        }
    }
    if (g == 0 && writer) {
#pragma unroll
        for (int j = 0; j < kHL; ++j)
            if (hbase + j < G) {
                sm.u.red.ml[warp][hbase + j][0] = M[j];
                sm.u.red.ml[warp][hbase + j][1] = Sl[j];
            }
    }
    __syncthreads();
    const int d = threadIdx.x;
    const size_t rec = u * p.nsplit + split;
#pragma unroll
    for (int gq = 0; gq < G; ++gq) {
        float m = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps4; ++w) m = fmaxf(m, sm.u.red.ml[w][gq][0]);
        float s_sum = 0.0f, a = 0.0f;
        if (m != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps4; ++w) {
                const float f = ex2_approx(sm.u.red.ml[w][gq][0] - m);
                s_sum = fmaf(sm.u.red.ml[w][gq][1], f, s_sum);
                a = fmaf(sm.u.red.acc[w][gq][d], f, a);
            }
        }
        p.ws_acc[(rec * G + gq) * kHD + d] = a;
        if (d == 0) {
            p.ws_ml[(rec * G + gq) * 2 + 0] = m;
            p.ws_ml[(rec * G + gq) * 2 + 1] = s_sum;
        }
    }
}

}  // namespace

// Splits: as many CTAs as are resident at once (one wave), within the record
// budget of the decode workspace (kMaxCtas + units records).  The kernel
// divides each unit's own length among its nsplit splits; split_tokens is
// the split length of a unit that fills the table.
bool make_int4_plan(int batch, int nkv, int max_blocks, int resident_ctas, int *nsplit, int *split_tokens) {
    const int64_t units = (int64_t)batch * nkv;
    if (units <= 0 || max_blocks <= 0) return false;
    const int64_t cap_tokens = (int64_t)max_blocks * kBS;
    int64_t ns = resident_ctas > 0 ? resident_ctas / units : 1;
    ns = ns < 1 ? 1 : ns;
    ns = ns > 1 + kMaxCtas / units ? 1 + kMaxCtas / units : ns;
    int64_t st = (cap_tokens + ns - 1) / ns;
    st = (st + kChunk4 - 1) / kChunk4 * kChunk4;
    *split_tokens = (int)st;
    *nsplit = (int)((cap_tokens + st - 1) / st);
    return true;
}

template <int G>
cudaError_t int4_occupancy(int *per) {
    cudaError_t e = cudaFuncSetAttribute(int4_decode_split_kernel<G, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Int4Smem<G>));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per, int4_decode_split_kernel<G, false>, kWarps4 * 32,
                                                         sizeof(Int4Smem<G>));
}

// CTAs of the decode kernel for G that the device holds at once.
int int4_resident_ctas(int group) {
    static int cached[64][9] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || group < 1 || group > 8) return 0;
    if (cached[dev][group] == 0) {
        int sms = 0, per = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cudaError_t e = cudaErrorInvalidValue;
        switch (group) {
            case 1: e = int4_occupancy<1>(&per); break;
            case 2: e = int4_occupancy<2>(&per); break;
            case 4: e = int4_occupancy<4>(&per); break;
            case 8: e = int4_occupancy<8>(&per); break;
            default: break;
        }
        if (e != cudaSuccess) return 0;
        cached[dev][group] = sms * per;
    }
    return cached[dev][group];
}

cudaError_t launch_int4_requantize(const Int4RequantParams &p, cudaStream_t s) {
    dim3 grid(p.max_count, p.nkv, p.batch);
    int4_requantize_kernel<<<grid, kReqWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_int4_append(const Int4AppendParams &p, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.n_new + kAppendWarps4 - 1) / kAppendWarps4, p.nkv, p.batch);
    cfg.blockDim = dim3(kAppendWarps4 * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, int4_append_kernel, p);
}

template <int G, bool kStep>
cudaError_t launch_int4_split_gs(const Int4DecodeParams &p, cudaStream_t s) {
    constexpr size_t smem = sizeof(Int4Smem<G>);
    static std::atomic<uint64_t> configured{0};
    return launch_after_setting(
        configured,
        [] {
            // the largest shared-memory carveout: in a mixed-precision decode the
            // int8 split joins an SM while one of these CTAs still runs there
            cudaError_t e = cudaFuncSetAttribute(int4_decode_split_kernel<G, kStep>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            return cudaFuncSetAttribute(int4_decode_split_kernel<G, kStep>,
                                        cudaFuncAttributePreferredSharedMemoryCarveout,
                                        (int)cudaSharedmemCarveoutMaxShared);
        },
        [&] {
            // a programmatic dependent of the previous kernel in the stream: every
            // thread waits for that kernel first (its outputs may be this
            // kernel's inputs, and a merge kernel before it may still read the
            // workspace), but the launch itself overlaps its end
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(p.nsplit, p.nkv, p.batch);
            cfg.blockDim = dim3(kWarps4 * 32);
            cfg.dynamicSmemBytes = smem;
            cfg.stream = s;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            return cudaLaunchKernelEx(&cfg, int4_decode_split_kernel<G, kStep>, p);
        });
}

template <int G>
cudaError_t launch_int4_split_g(const Int4DecodeParams &p, cudaStream_t s) {
    return p.k_new ? launch_int4_split_gs<G, true>(p, s) : launch_int4_split_gs<G, false>(p, s);
}

cudaError_t launch_int4_decode_split(const Int4DecodeParams &p, int group, cudaStream_t s) {
    switch (group) {
        case 1: return launch_int4_split_g<1>(p, s);
        case 2: return launch_int4_split_g<2>(p, s);
        case 4: return launch_int4_split_g<4>(p, s);
        case 8: return launch_int4_split_g<8>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvq8
