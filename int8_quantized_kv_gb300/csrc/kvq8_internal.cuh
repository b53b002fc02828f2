// kvq8_internal.cuh -- declarations shared by the translation units of libkvq8
// (kernel launchers, the decode plan, device helpers).  Not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "kvq8.h"

namespace kvq8 {

// Runs `launch` after `set` (a kernel attribute such as its dynamic shared-
// memory limit) has been applied once on the current device: the setting
// belongs to the device's context, and applying it on every launch costs a
// driver call per launch.  `configured` holds one bit per device.  Should a
// launch be refused as an invalid configuration although the bit is set (the
// context was re-created since), the attribute is applied again and the
// launch repeated once.  `launch` returns that launch's own status
// (cudaLaunchKernelEx), so nothing runs twice.
template <typename SetFn, typename LaunchFn>
cudaError_t launch_after_setting(std::atomic<uint64_t> &configured, SetFn set, LaunchFn launch) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
    cudaError_t e;
    if (bit == 0 || !(configured.load(std::memory_order_relaxed) & bit)) {
        if ((e = set()) != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_relaxed);
        return launch();
    }
    if ((e = launch()) != cudaErrorInvalidValue) return e;
    (void)cudaGetLastError();
    if ((e = set()) != cudaSuccess) return e;
    return launch();
}

constexpr int kHD = 128;           // head dimension
constexpr int kBS = 256;           // tokens per cache block
constexpr int kQB = 32;            // query quantisation block
constexpr int kNQB = kHD / kQB;    // query blocks per head
constexpr int kMaxGridYZ = 65535;  // launch limit on gridDim.y / gridDim.z

// ----------------------------------------------------------------- append --
struct AppendParams {
    const float *k_new, *v_new;   // [batch][n_new][nkv][hd]
    int batch, n_new, nkv;
    const int32_t *start_pos;     // [batch]: position of each sequence's first new token
    const int32_t *block_table;   // [batch][max_blocks]
    int max_blocks, num_blocks;
    int8_t *k_pool, *v_pool;
    float *k_scale, *v_scale;
    uint32_t *dev_status;
};
cudaError_t launch_quantize_append(const AppendParams &p, cudaStream_t s);
cudaError_t launch_quantize_q(const float *q, int64_t n_rows, int8_t *codes,
                              float *scales, cudaStream_t s);

// ----------------------------------------------------------------- decode --
// Cache tile geometry.  One (block, kv head) tile holds 256 tokens:
//   K: [256 tokens][128 B]; the 16-byte chunk j of token row t is stored at
//      chunk position j ^ (t & 7), so lanes reading one row each hit distinct
//      shared-memory banks after a plain copy.
//   V: [4 quarters][128 dims][64 B]: dim-major per 64-token quarter.
// A 64-token window of a tile (a decode "stage") is therefore four contiguous
// runs: 8 KiB of K, 8 KiB of V and 256 B of each scale array.
constexpr int kStageTok = 64;
constexpr int kStageKBytes = kStageTok * kHD;     // 8192
constexpr int kStageVBytes = kHD * kStageTok;     // 8192
constexpr int kStageSBytes = kStageTok * 4;       // 256
constexpr int kStageBytes = kStageKBytes + kStageVBytes + 2 * kStageSBytes;
constexpr int kTileVQuarter = kHD * kStageTok;    // bytes of one V quarter
constexpr int kMaxCtas = 1024;                    // upper bound of the split grid

// Split-KV plan: the split kernel runs one persistent CTA per SM; the global
// sequence of 64-token stages (units in order (sequence, kv head)) is cut into
// equal contiguous ranges, one per CTA.  A (CTA c, unit u) segment writes
// partial record c + u; meta[u] names the first CTA of unit u and its count.
struct DecodePlan {
    int group;          // G = nqh / nkv
    int64_t units;      // batch * nkv
    int64_t records;    // kMaxCtas + units
    size_t meta_offset, ml_offset, acc_offset, bytes;  // workspace layout
};
bool make_decode_plan(int batch, int nqh, int nkv, int max_blocks, DecodePlan *plan);

struct DecodeParams {
    const float *q;               // [batch][nqh][hd]
    int batch, nqh, nkv;
    const int8_t *k_pool, *v_pool;
    const float *k_scale, *v_scale;
    int num_blocks;
    const int32_t *block_table;
    int max_blocks;
    const int32_t *ctx_lens;
    float sm_scale_log2;          // sm_scale * log2(e): softmax runs in base 2
    // A decode step's new token ([batch][nkv][hd] each; null otherwise): the
    // split kernel quantises it into position ctx_lens[b] - 1, in the stage it
    // copies and in the pools, which are then the caller's writable buffers
    const float *k_new, *v_new;
    int2 *ws_meta;                // [units]: (first CTA, CTA count)
    float *ws_ml;                 // [records][G][2]  (running max M, sum S)
    float *ws_acc;                // [records][G][hd] (unnormalised V accumulator)
    uint32_t *dev_status;
    float *out;                   // [batch][nqh][hd] (combine only)
    // mixed precision by token age (null otherwise): the int8 part starts at
    // block first_q8_block[b]; the combine also merges the 4-bit split's records
    const int32_t *first_q8_block;
    const int2 *ws_meta2;
    const float *ws_ml2, *ws_acc2;
    // Nonzero: the cache, block_table and ctx_lens were final before the
    // kernel preceding this call in the stream began, so the split kernel's
    // prologue and copies run before it waits for that kernel (only q, k_new,
    // v_new and the workspace wait).  Zero: every thread waits first.
    int cache_ready;
};
cudaError_t launch_decode_split(const DecodeParams &p, int group, cudaStream_t s);
cudaError_t launch_decode_combine(const DecodeParams &p, int group, cudaStream_t s);
// The merge of the 4-bit decode: unit u's records are u * nsplit + j for its
// int4_split_count(L, nsplit) splits j (nsplit <= 8), read without the record
// directory.
cudaError_t launch_decode_combine_fixed(const DecodeParams &p, int group, int nsplit, cudaStream_t s);

// ------------------------------------------------------------ INT4 cache --
// A unit of L tokens cut into nsplit splits of whole 32-token chunks (the
// 4-bit decode): tokens per split, and how many splits hold tokens.
__host__ __device__ inline int int4_split_tokens(int L, int nsplit) {
    const int st = ((L + nsplit - 1) / nsplit + 31) / 32 * 32;
    return st > 32 ? st : 32;
}
__host__ __device__ inline int int4_split_count(int L, int nsplit) {
    const int st = int4_split_tokens(L, nsplit);
    return (L + st - 1) / st;
}

struct Int4AppendParams {
    const float *k_new, *v_new;   // [batch][n_new][nkv][hd]
    int batch, n_new, nkv;
    const int32_t *start_pos;     // [batch]
    const int32_t *block_table;
    int max_blocks, num_blocks;
    uint8_t *k_codes, *v_codes;   // [num_blocks][nkv][256][64]
    float *k_param, *v_param;     // [num_blocks][nkv][256][4]
    uint32_t *dev_status;
};

struct Int4DecodeParams {
    const float *q;               // [batch][nqh][hd]
    // A decode step's new token ([batch][nkv][hd] each; null otherwise): the
    // split kernel quantises it into position ctx_lens[b] - 1, in the chunk it
    // stages and in the cache, which is then the caller's writable buffer
    const float *k_new, *v_new;
    const int32_t *n4_blocks;     // null, or: only tokens [0, 256 * n4_blocks[b]) (mixed precision)
    int batch, nqh, nkv;
    const uint8_t *k_codes, *v_codes;
    const float *k_param, *v_param;
    int num_blocks;
    const int32_t *block_table;
    int max_blocks;
    const int32_t *ctx_lens;
    float sm_scale_log2;
    int nsplit, split_tokens;     // unit u's split j writes record u*nsplit + j
    int2 *ws_meta;
    float *ws_ml, *ws_acc;        // same record format as DecodeParams
    uint32_t *dev_status;
};
// Mixed precision by token age: logical blocks [blk_from[b], blk_to[b]) of
// sequence b are requantised from the int8 tiles table8[b][j] into the 4-bit
// tiles table4[b][j].
struct Int4RequantParams {
    int batch, nkv;
    const int8_t *k_pool, *v_pool;
    const float *k_scale, *v_scale;
    int num_blocks8;
    const int32_t *table8;
    uint8_t *k_codes, *v_codes;
    float *k_param, *v_param;
    int num_blocks4;
    const int32_t *table4;
    int max_blocks;
    const int32_t *blk_from, *blk_to;
    int max_count;                // grid bound: blk_to - blk_from <= max_count
    uint32_t *dev_status;
};
cudaError_t launch_int4_requantize(const Int4RequantParams &p, cudaStream_t s);
bool make_int4_plan(int batch, int nkv, int max_blocks, int resident_ctas, int *nsplit, int *split_tokens);
int int4_resident_ctas(int group);
cudaError_t launch_int4_append(const Int4AppendParams &p, cudaStream_t s);
cudaError_t launch_int4_decode_split(const Int4DecodeParams &p, int group, cudaStream_t s);

// ------------------------------------------------------------ fp32 cache --
struct F32AppendParams {
    const float *k_new, *v_new;   // [batch][n_new][nkv][hd]
    int batch, n_new, nkv;
    const int32_t *start_pos;     // [batch]
    const int32_t *block_table;
    int max_blocks, num_blocks;
    float *k_cache, *v_cache;     // [num_blocks][nkv][256][hd]
    uint32_t *dev_status;
};

struct F32DecodeParams {
    const float *q;               // [batch][nqh][hd]
    int batch, nqh, nkv;
    const float *k_cache, *v_cache;
    int num_blocks;
    const int32_t *block_table;
    int max_blocks;
    const int32_t *ctx_lens;
    float sm_scale_log2;
    int nsplit, split_tokens;     // unit u's split j writes record u*nsplit + j
    int2 *ws_meta;
    float *ws_ml, *ws_acc;        // same record format as DecodeParams
    uint32_t *dev_status;
};
bool make_f32_plan(int batch, int nkv, int max_blocks, int *nsplit, int *split_tokens);
cudaError_t launch_f32_append(const F32AppendParams &p, cudaStream_t s);
cudaError_t launch_f32_decode_split(const F32DecodeParams &p, int group, cudaStream_t s);

// One warp waiting, bounded by timeout_ns, on an mbarrier phase that nothing
// completes (kvq8_selftest_bounded_wait).
cudaError_t launch_bounded_wait_selftest(uint32_t *dev_status, uint64_t timeout_ns, unsigned long long *waited_ns,
                                         cudaStream_t s);

}  // namespace kvq8
