// noalloc.cu -- kvq8_decode_attn_noalloc: the decode of kvq8_decode_attn for
// callers that cannot allocate device memory.
//
// Some callers are handed only their input and output buffers and a stream:
// plugin hosts that own the device allocator, code paths where a cudaMalloc
// would synchronise the device or is not permitted at all.  They cannot
// provide the workspace that holds the split-KV partial results, so this entry
// point keeps that scratch in a file-scope static device array instead.  The
// array exists once per device in every process that loads the library and
// lives until the process exits.  Nothing here allocates: no cudaMalloc, no
// cudaFree, no allocating library routine.
#include <mutex>

#include "kvq8_internal.cuh"

namespace {

// Scratch for the split-KV partial records (running max, softmax sum and V
// accumulator per split and query head).
static __device__ __align__(256) unsigned char g_decode_scratch[KVQ8_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices];  // device address of g_decode_scratch, per device

// In host code g_decode_scratch names a host-side shadow, not device memory;
// the kernels must be given the address the runtime reports for the current
// device.  Looked up once per device, with that device current, on the first
// call that reaches the kernels; the address belongs to the device's context
// of that moment (a cudaDeviceReset discards it, see kvq8.h).
kvq8_status scratch_for_current_device(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVQ8_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KVQ8_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
            return KVQ8_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return KVQ8_OK;
}

}  // namespace

extern "C" kvq8_status kvq8_decode_attn_noalloc(
    const float *q, int batch, int nqh, int nkv, int hd, const int8_t *k_pool,
    const int8_t *v_pool, const float *k_scale, const float *v_scale, int num_blocks,
    const int32_t *block_table, int max_blocks, int block_size, const int32_t *ctx_lens,
    float sm_scale, float *out, uint32_t *dev_status, void *stream) {
    // Every argument check of kvq8_decode_attn, in its order: called without a
    // workspace it returns before enqueuing anything -- an argument error, OK
    // for an empty batch, or KVQ8_ERR_WORKSPACE once everything else is valid.
    kvq8_status st = kvq8_decode_attn(q, batch, nqh, nkv, hd, k_pool, v_pool, k_scale, v_scale,
                                      num_blocks, block_table, max_blocks, block_size, ctx_lens,
                                      sm_scale, out, nullptr, 0, dev_status, stream);
    if (st != KVQ8_ERR_WORKSPACE) return st;
    const size_t need =
        kvq8_decode_workspace_bytes(batch, nqh, nkv, hd, max_blocks, block_size);
    if (need == 0 || need > (size_t)KVQ8_NOALLOC_SCRATCH_BYTES) return KVQ8_ERR_WORKSPACE;
    void *scratch = nullptr;
    if ((st = scratch_for_current_device(&scratch)) != KVQ8_OK) return st;
    return kvq8_decode_attn(q, batch, nqh, nkv, hd, k_pool, v_pool, k_scale, v_scale, num_blocks,
                            block_table, max_blocks, block_size, ctx_lens, sm_scale, out, scratch,
                            (size_t)KVQ8_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
