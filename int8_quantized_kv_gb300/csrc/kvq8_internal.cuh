// kvq8_internal.cuh -- declarations shared by the translation units of libkvq8
// (kernel launchers, the decode plan, device helpers).  Not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq8.h"

namespace kvq8 {

constexpr int kHD = 128;           // head dimension
constexpr int kBS = 256;           // tokens per cache block
constexpr int kQB = 32;            // query quantisation block
constexpr int kNQB = kHD / kQB;    // query blocks per head
constexpr int kMaxGridYZ = 65535;  // launch limit on gridDim.y / gridDim.z

// ----------------------------------------------------------------- append --
struct AppendParams {
    const float *k_new, *v_new;   // [batch][n_new][nkv][hd]
    int batch, n_new, nkv;
    const int32_t *start_pos;     // [batch]
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
// Split-KV plan: every (sequence, kv head) unit is cut into splits of
// split_blocks cache blocks; a split writes one partial record per query head.
struct DecodePlan {
    int group;          // G = nqh / nkv
    int split_blocks;   // cache blocks per split
    int nsplit;         // splits per unit (covering max_blocks blocks)
    int64_t records;    // batch * nkv * nsplit
    size_t ml_offset, acc_offset, bytes;  // workspace layout
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
    float *ws_ml;                 // [records][G][2]  (running max M, sum S)
    float *ws_acc;                // [records][G][hd] (unnormalised V accumulator)
    int nsplit, split_blocks;
    uint32_t *dev_status;
    float *out;                   // [batch][nqh][hd] (combine only)
};
cudaError_t launch_decode_split(const DecodeParams &p, int group, cudaStream_t s);
cudaError_t launch_decode_combine(const DecodeParams &p, int group, cudaStream_t s);

}  // namespace kvq8
