// abi.cu -- the extern "C" entry points of libkvq8 (declared in kvq8.h):
// argument validation, workspace layout and kernel launches.  No allocation,
// no synchronisation: every call enqueues on the caller's stream.
#include <math.h>

#include "kvq8_internal.cuh"

using namespace kvq8;

namespace {

bool aligned(const void *ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

kvq8_status check_shape(int hd, int block_size) {
    if (hd != kHD || block_size != kBS) return KVQ8_ERR_UNSUPPORTED;
    return KVQ8_OK;
}

kvq8_status check_heads(int nqh, int nkv) {
    if (nqh <= 0 || nkv <= 0) return KVQ8_ERR_INVALID_ARG;
    if (nqh % nkv) return KVQ8_ERR_UNSUPPORTED;
    const int G = nqh / nkv;
    if (G != 1 && G != 2 && G != 4 && G != 8) return KVQ8_ERR_UNSUPPORTED;
    if (nkv > kMaxGridYZ || nqh > 2147483647 / kHD) return KVQ8_ERR_UNSUPPORTED;
    return KVQ8_OK;
}

// Shared validation of the decode entry points (pool and table arguments).
kvq8_status check_decode_args(const float *q, int batch, int nqh, int nkv, int hd,
                              const int8_t *k_pool, const int8_t *v_pool, const float *k_scale,
                              const float *v_scale, int num_blocks, const int32_t *block_table,
                              int max_blocks, int block_size, const int32_t *ctx_lens) {
    kvq8_status st = check_shape(hd, block_size);
    if (st != KVQ8_OK) return st;
    if ((st = check_heads(nqh, nkv)) != KVQ8_OK) return st;
    if (batch < 0 || num_blocks <= 0 || max_blocks <= 0) return KVQ8_ERR_INVALID_ARG;
    if (max_blocks > 2147483647 / kBS) return KVQ8_ERR_UNSUPPORTED;
    if (batch > kMaxGridYZ) return KVQ8_ERR_UNSUPPORTED;
    if (batch == 0) return KVQ8_OK;
    if (!q || !k_pool || !v_pool || !k_scale || !v_scale || !block_table || !ctx_lens)
        return KVQ8_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
        !aligned(k_scale, 16) || !aligned(v_scale, 16) || !aligned(block_table, 4) ||
        !aligned(ctx_lens, 4))
        return KVQ8_ERR_INVALID_ARG;
    return KVQ8_OK;
}

kvq8_status fill_decode_params(const float *q, int batch, int nqh, int nkv,
                               const int8_t *k_pool, const int8_t *v_pool, const float *k_scale,
                               const float *v_scale, int num_blocks, const int32_t *block_table,
                               int max_blocks, const int32_t *ctx_lens, float sm_scale,
                               const void *workspace, size_t workspace_bytes,
                               uint32_t *dev_status, DecodeParams *p, DecodePlan *plan) {
    if (!make_decode_plan(batch, nqh, nkv, max_blocks, plan)) return KVQ8_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < plan->bytes)
        return KVQ8_ERR_WORKSPACE;
    char *ws = (char *)workspace;
    p->q = q;
    p->batch = batch;
    p->nqh = nqh;
    p->nkv = nkv;
    p->k_pool = k_pool;
    p->v_pool = v_pool;
    p->k_scale = k_scale;
    p->v_scale = v_scale;
    p->num_blocks = num_blocks;
    p->block_table = block_table;
    p->max_blocks = max_blocks;
    p->ctx_lens = ctx_lens;
    p->sm_scale_log2 = sm_scale * 1.4426950408889634f;
    p->k_new = nullptr;
    p->v_new = nullptr;
    p->ws_meta = (int2 *)(ws + plan->meta_offset);
    p->ws_ml = (float *)(ws + plan->ml_offset);
    p->ws_acc = (float *)(ws + plan->acc_offset);
    p->dev_status = dev_status;
    p->out = nullptr;
    p->first_q8_block = nullptr;
    p->cache_ready = 0;
    p->ws_meta2 = nullptr;
    p->ws_ml2 = nullptr;
    p->ws_acc2 = nullptr;
    return KVQ8_OK;
}

}  // namespace

extern "C" {

const char *kvq8_status_str(int status) {
    switch (status) {
        case KVQ8_OK: return "KVQ8_OK";
        case KVQ8_ERR_INVALID_ARG: return "KVQ8_ERR_INVALID_ARG";
        case KVQ8_ERR_UNSUPPORTED: return "KVQ8_ERR_UNSUPPORTED";
        case KVQ8_ERR_WORKSPACE: return "KVQ8_ERR_WORKSPACE";
        case KVQ8_ERR_CUDA: return "KVQ8_ERR_CUDA";
        default: return "KVQ8_UNKNOWN_STATUS";
    }
}

int kvq8_abi_version(void) { return 1; }

size_t kvq8_kv_pool_bytes(int num_blocks, int nkv, int hd, int block_size) {
    if (num_blocks < 0 || nkv < 0 || hd < 0 || block_size < 0) return 0;
    return (size_t)num_blocks * nkv * block_size * hd;
}

size_t kvq8_scale_pool_bytes(int num_blocks, int nkv, int block_size) {
    if (num_blocks < 0 || nkv < 0 || block_size < 0) return 0;
    return (size_t)num_blocks * nkv * block_size * sizeof(float);
}

size_t kvq8_cache_bytes_per_token(int nkv, int hd) {
    if (nkv < 0 || hd < 0) return 0;
    return (size_t)nkv * (2 * (size_t)hd + 2 * sizeof(float));
}

// Checks the arguments of kvq8_quantize_append and fills p; *noop when there
// is nothing to append.
static kvq8_status prepare_append(const float *k_new, const float *v_new, int batch, int n_new, int nkv,
                                  int hd, const int32_t *start_pos, const int32_t *block_table,
                                  int max_blocks, int block_size, int num_blocks, int8_t *k_pool,
                                  int8_t *v_pool, float *k_scale, float *v_scale, uint32_t *dev_status,
                                  AppendParams *p, bool *noop) {
    *noop = true;
    kvq8_status st = check_shape(hd, block_size);
    if (st != KVQ8_OK) return st;
    if (batch < 0 || n_new < 0 || nkv <= 0 || num_blocks <= 0 || max_blocks <= 0)
        return KVQ8_ERR_INVALID_ARG;
    if (max_blocks > 2147483647 / kBS) return KVQ8_ERR_UNSUPPORTED;
    if (batch > kMaxGridYZ || nkv > kMaxGridYZ) return KVQ8_ERR_UNSUPPORTED;
    if (batch == 0 || n_new == 0) return KVQ8_OK;
    if (!k_new || !v_new || !start_pos || !block_table || !k_pool || !v_pool || !k_scale ||
        !v_scale)
        return KVQ8_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pool, 16) ||
        !aligned(v_pool, 16) || !aligned(k_scale, 16) || !aligned(v_scale, 16) ||
        !aligned(start_pos, 4) || !aligned(block_table, 4))
        return KVQ8_ERR_INVALID_ARG;
    p->k_new = k_new;
    p->v_new = v_new;
    p->batch = batch;
    p->n_new = n_new;
    p->nkv = nkv;
    p->start_pos = start_pos;
    p->block_table = block_table;
    p->max_blocks = max_blocks;
    p->num_blocks = num_blocks;
    p->k_pool = k_pool;
    p->v_pool = v_pool;
    p->k_scale = k_scale;
    p->v_scale = v_scale;
    p->dev_status = dev_status;
    *noop = false;
    return KVQ8_OK;
}

// The device address of host memory that the GPU can access directly and that
// is 16-byte aligned there: page-locked memory mapped into the device's
// address space (with unified addressing, every page-locked allocation);
// null for anything else (pageable or device memory), which the caller then
// copies.
static const void *mapped_host(const void *h) {
    if (!h || !aligned(h, 16)) return nullptr;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
        (void)cudaGetLastError();   // an unknown pointer: not mapped
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr || !aligned(a.devicePointer, 16))
        return nullptr;
    return a.devicePointer;
}

// One asynchronous copy (a no-op for 0 bytes).
static bool copy_async(void *dst, const void *src, size_t bytes, cudaMemcpyKind kind, cudaStream_t s) {
    return bytes == 0 || cudaMemcpyAsync(dst, src, bytes, kind, s) == cudaSuccess;
}

kvq8_status kvq8_quantize_append(const float *k_new, const float *v_new, int batch, int n_new,
                                 int nkv, int hd, const int32_t *start_pos,
                                 const int32_t *block_table, int max_blocks, int block_size,
                                 int num_blocks, int8_t *k_pool, int8_t *v_pool, float *k_scale,
                                 float *v_scale, uint32_t *dev_status, void *stream) {
    AppendParams p;
    bool noop;
    const kvq8_status st = prepare_append(k_new, v_new, batch, n_new, nkv, hd, start_pos, block_table,
                                          max_blocks, block_size, num_blocks, k_pool, v_pool, k_scale,
                                          v_scale, dev_status, &p, &noop);
    if (st != KVQ8_OK || noop) return st;
    if (launch_quantize_append(p, (cudaStream_t)stream) != cudaSuccess) return KVQ8_ERR_CUDA;
    return KVQ8_OK;
}

kvq8_status kvq8_quantize_append_host(const float *k_new_host, const float *v_new_host,
                                      float *k_new, float *v_new, int batch, int n_new, int nkv,
                                      int hd, const int32_t *start_pos, const int32_t *block_table,
                                      int max_blocks, int block_size, int num_blocks, int8_t *k_pool,
                                      int8_t *v_pool, float *k_scale, float *v_scale,
                                      uint32_t *dev_status, void *stream) {
    AppendParams p;
    bool noop;
    const kvq8_status st = prepare_append(k_new, v_new, batch, n_new, nkv, hd, start_pos, block_table,
                                          max_blocks, block_size, num_blocks, k_pool, v_pool, k_scale,
                                          v_scale, dev_status, &p, &noop);
    if (st != KVQ8_OK || noop) return st;
    if (!k_new_host || !v_new_host) return KVQ8_ERR_INVALID_ARG;
    const size_t bytes = (size_t)batch * n_new * nkv * hd * sizeof(float);
    cudaStream_t s = (cudaStream_t)stream;
    if (!copy_async(k_new, k_new_host, bytes, cudaMemcpyHostToDevice, s) ||
        !copy_async(v_new, v_new_host, bytes, cudaMemcpyHostToDevice, s))
        return KVQ8_ERR_CUDA;
    if (launch_quantize_append(p, s) != cudaSuccess) return KVQ8_ERR_CUDA;
    return KVQ8_OK;
}

kvq8_status kvq8_quantize_q(const float *q, int64_t n_rows, int hd, int8_t *q_codes,
                            float *q_scales, void *stream) {
    if (hd != kHD) return KVQ8_ERR_UNSUPPORTED;
    if (n_rows < 0) return KVQ8_ERR_INVALID_ARG;
    if (n_rows > (int64_t)4 * 2147483647) return KVQ8_ERR_UNSUPPORTED;
    if (n_rows == 0) return KVQ8_OK;
    if (!q || !q_codes || !q_scales || !aligned(q, 4) || !aligned(q_scales, 4))
        return KVQ8_ERR_INVALID_ARG;
    if (launch_quantize_q(q, n_rows, q_codes, q_scales, (cudaStream_t)stream) != cudaSuccess)
        return KVQ8_ERR_CUDA;
    return KVQ8_OK;
}

size_t kvq8_decode_workspace_bytes(int batch, int nqh, int nkv, int hd, int max_blocks,
                                   int block_size) {
    if (check_shape(hd, block_size) != KVQ8_OK || check_heads(nqh, nkv) != KVQ8_OK) return 0;
    DecodePlan plan;
    if (!make_decode_plan(batch, nqh, nkv, max_blocks, &plan)) return 0;
    return plan.bytes;
}

kvq8_status kvq8_decode_split(const float *q, int batch, int nqh, int nkv, int hd,
                              const int8_t *k_pool, const int8_t *v_pool, const float *k_scale,
                              const float *v_scale, int num_blocks, const int32_t *block_table,
                              int max_blocks, int block_size, const int32_t *ctx_lens,
                              float sm_scale, void *workspace, size_t workspace_bytes,
                              uint32_t *dev_status, void *stream) {
    kvq8_status st = check_decode_args(q, batch, nqh, nkv, hd, k_pool, v_pool, k_scale, v_scale,
                                       num_blocks, block_table, max_blocks, block_size, ctx_lens);
    if (st != KVQ8_OK || batch == 0) return st;
    if (!isfinite(sm_scale)) return KVQ8_ERR_INVALID_ARG;
    DecodeParams p;
    DecodePlan plan;
    st = fill_decode_params(q, batch, nqh, nkv, k_pool, v_pool, k_scale, v_scale, num_blocks,
                            block_table, max_blocks, ctx_lens, sm_scale, workspace,
                            workspace_bytes, dev_status, &p, &plan);
    if (st != KVQ8_OK) return st;
    if (launch_decode_split(p, plan.group, (cudaStream_t)stream) != cudaSuccess)
        return KVQ8_ERR_CUDA;
    return KVQ8_OK;
}

kvq8_status kvq8_decode_combine(int batch, int nqh, int nkv, int hd, int max_blocks,
                                int block_size, const int32_t *ctx_lens, const void *workspace,
                                size_t workspace_bytes, float *out, void *stream) {
    kvq8_status st = check_shape(hd, block_size);
    if (st != KVQ8_OK) return st;
    if ((st = check_heads(nqh, nkv)) != KVQ8_OK) return st;
    if (batch < 0 || max_blocks <= 0) return KVQ8_ERR_INVALID_ARG;
    if (max_blocks > 2147483647 / kBS) return KVQ8_ERR_UNSUPPORTED;
    if (batch > kMaxGridYZ) return KVQ8_ERR_UNSUPPORTED;
    if (batch == 0) return KVQ8_OK;
    if (!ctx_lens || !out || !aligned(out, 16) || !aligned(ctx_lens, 4))
        return KVQ8_ERR_INVALID_ARG;
    DecodeParams p;
    DecodePlan plan;
    st = fill_decode_params(nullptr, batch, nqh, nkv, nullptr, nullptr, nullptr, nullptr, 1,
                            nullptr, max_blocks, ctx_lens, 1.0f, workspace, workspace_bytes,
                            nullptr, &p, &plan);
    if (st != KVQ8_OK) return st;
    p.out = out;
    if (launch_decode_combine(p, plan.group, (cudaStream_t)stream) != cudaSuccess)
        return KVQ8_ERR_CUDA;
    return KVQ8_OK;
}

kvq8_status kvq8_decode_attn(const float *q, int batch, int nqh, int nkv, int hd,
                             const int8_t *k_pool, const int8_t *v_pool, const float *k_scale,
                             const float *v_scale, int num_blocks, const int32_t *block_table,
                             int max_blocks, int block_size, const int32_t *ctx_lens,
                             float sm_scale, float *out, void *workspace, size_t workspace_bytes,
                             uint32_t *dev_status, void *stream) {
    kvq8_status st = check_decode_args(q, batch, nqh, nkv, hd, k_pool, v_pool, k_scale, v_scale,
                                       num_blocks, block_table, max_blocks, block_size, ctx_lens);
    if (st != KVQ8_OK || batch == 0) return st;
    if (!out || !aligned(out, 16) || !isfinite(sm_scale)) return KVQ8_ERR_INVALID_ARG;
    DecodeParams p;
    DecodePlan plan;
    st = fill_decode_params(q, batch, nqh, nkv, k_pool, v_pool, k_scale, v_scale, num_blocks,
                            block_table, max_blocks, ctx_lens, sm_scale, workspace,
                            workspace_bytes, dev_status, &p, &plan);
    if (st != KVQ8_OK) return st;
    p.out = out;
    cudaStream_t s = (cudaStream_t)stream;
    if (launch_decode_split(p, plan.group, s) != cudaSuccess) return KVQ8_ERR_CUDA;
    if (launch_decode_combine(p, plan.group, s) != cudaSuccess) return KVQ8_ERR_CUDA;
    return KVQ8_OK;
}

// Checks the arguments of kvq8_decode_step and fills the parameters of its
// two launches (the split kernel also appends the step's new token).
static kvq8_status prepare_decode_step(const float *q, const float *k_new, const float *v_new, int batch,
                                       int nqh, int nkv, int hd, int8_t *k_pool, int8_t *v_pool,
                                       float *k_scale, float *v_scale, int num_blocks,
                                       const int32_t *block_table, int max_blocks, int block_size,
                                       const int32_t *ctx_lens, float sm_scale, float *out,
                                       void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                                       DecodeParams *p, DecodePlan *plan) {
    kvq8_status st = check_decode_args(q, batch, nqh, nkv, hd, k_pool, v_pool, k_scale, v_scale,
                                       num_blocks, block_table, max_blocks, block_size, ctx_lens);
    if (st != KVQ8_OK || batch == 0) return st;
    if (!out || !aligned(out, 16) || !isfinite(sm_scale)) return KVQ8_ERR_INVALID_ARG;
    if (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16)) return KVQ8_ERR_INVALID_ARG;
    st = fill_decode_params(q, batch, nqh, nkv, k_pool, v_pool, k_scale, v_scale, num_blocks,
                            block_table, max_blocks, ctx_lens, sm_scale, workspace,
                            workspace_bytes, dev_status, p, plan);
    if (st != KVQ8_OK) return st;
    p->out = out;
    p->k_new = k_new;   // appended at ctx_lens[b] - 1 by the split kernel
    p->v_new = v_new;
    return KVQ8_OK;
}

static kvq8_status launch_decode_step(const DecodeParams &p, const DecodePlan &plan, cudaStream_t s) {
    if (launch_decode_split(p, plan.group, s) != cudaSuccess) return KVQ8_ERR_CUDA;
    if (launch_decode_combine(p, plan.group, s) != cudaSuccess) return KVQ8_ERR_CUDA;
    return KVQ8_OK;
}

kvq8_status kvq8_decode_step(const float *q, const float *k_new, const float *v_new, int batch,
                             int nqh, int nkv, int hd, int8_t *k_pool, int8_t *v_pool,
                             float *k_scale, float *v_scale, int num_blocks,
                             const int32_t *block_table, int max_blocks, int block_size,
                             const int32_t *ctx_lens, float sm_scale, float *out, void *workspace,
                             size_t workspace_bytes, uint32_t *dev_status, void *stream) {
    DecodeParams p;
    DecodePlan plan;
    const kvq8_status st = prepare_decode_step(q, k_new, v_new, batch, nqh, nkv, hd, k_pool, v_pool, k_scale,
                                               v_scale, num_blocks, block_table, max_blocks, block_size,
                                               ctx_lens, sm_scale, out, workspace, workspace_bytes,
                                               dev_status, &p, &plan);
    if (st != KVQ8_OK || batch == 0) return st;
    return launch_decode_step(p, plan, (cudaStream_t)stream);
}

kvq8_status kvq8_decode_step_ex(const float *q, const float *k_new, const float *v_new, int batch,
                                int nqh, int nkv, int hd, int8_t *k_pool, int8_t *v_pool,
                                float *k_scale, float *v_scale, int num_blocks,
                                const int32_t *block_table, int max_blocks, int block_size,
                                const int32_t *ctx_lens, float sm_scale, float *out, void *workspace,
                                size_t workspace_bytes, uint32_t *dev_status, uint32_t flags,
                                void *stream) {
    if (flags & ~(uint32_t)KVQ8_STEP_CACHE_READY) return KVQ8_ERR_INVALID_ARG;
    DecodeParams p;
    DecodePlan plan;
    const kvq8_status st = prepare_decode_step(q, k_new, v_new, batch, nqh, nkv, hd, k_pool, v_pool, k_scale,
                                               v_scale, num_blocks, block_table, max_blocks, block_size,
                                               ctx_lens, sm_scale, out, workspace, workspace_bytes,
                                               dev_status, &p, &plan);
    if (st != KVQ8_OK || batch == 0) return st;
    p.cache_ready = (flags & KVQ8_STEP_CACHE_READY) ? 1 : 0;
    return launch_decode_step(p, plan, (cudaStream_t)stream);
}

kvq8_status kvq8_decode_step_host(const float *q_host, const float *k_new_host, const float *v_new_host,
                                  float *out_host, float *q, float *k_new, float *v_new, int batch,
                                  int nqh, int nkv, int hd, int8_t *k_pool, int8_t *v_pool,
                                  float *k_scale, float *v_scale, int num_blocks,
                                  const int32_t *block_table, int max_blocks, int block_size,
                                  const int32_t *ctx_lens, float sm_scale, float *out, void *workspace,
                                  size_t workspace_bytes, uint32_t *dev_status, void *stream) {
    DecodeParams p;
    DecodePlan plan;
    kvq8_status st = prepare_decode_step(q, k_new, v_new, batch, nqh, nkv, hd, k_pool, v_pool, k_scale,
                                         v_scale, num_blocks, block_table, max_blocks, block_size,
                                         ctx_lens, sm_scale, out, workspace, workspace_bytes, dev_status,
                                         &p, &plan);
    if (st != KVQ8_OK || batch == 0) return st;
    if (!q_host || !k_new_host || !v_new_host || !out_host) return KVQ8_ERR_INVALID_ARG;
    const size_t qbytes = (size_t)batch * nqh * hd * sizeof(float);
    const size_t kvbytes = (size_t)batch * nkv * hd * sizeof(float);
    cudaStream_t s = (cudaStream_t)stream;
    // Host buffers that the GPU can address (page-locked memory mapped into the
    // device's address space) are read and written by the kernels themselves:
    // no copy is queued and the step's two launches stay chained.
    const void *qm = mapped_host(q_host), *km = mapped_host(k_new_host), *vm = mapped_host(v_new_host);
    const void *om = mapped_host(out_host);
    if (qm && km && vm && om) {
        p.q = static_cast<const float *>(qm);
        p.k_new = static_cast<const float *>(km);
        p.v_new = static_cast<const float *>(vm);
        p.out = static_cast<float *>(const_cast<void *>(om));
        return launch_decode_step(p, plan, s);
    }
    if (!copy_async(q, q_host, qbytes, cudaMemcpyHostToDevice, s) ||
        !copy_async(k_new, k_new_host, kvbytes, cudaMemcpyHostToDevice, s) ||
        !copy_async(v_new, v_new_host, kvbytes, cudaMemcpyHostToDevice, s))
        return KVQ8_ERR_CUDA;
    st = launch_decode_step(p, plan, s);
    if (st != KVQ8_OK) return st;
    if (!copy_async(out_host, out, qbytes, cudaMemcpyDeviceToHost, s)) return KVQ8_ERR_CUDA;
    return KVQ8_OK;
}

const void *kvq8_host_device_pointer(const void *host_ptr) { return mapped_host(host_ptr); }

kvq8_status kvq8_selftest_bounded_wait(uint32_t *dev_status, uint64_t timeout_ns,
                                       unsigned long long *waited_ns, void *stream) {
    if (!dev_status || !aligned(dev_status, 4) || (waited_ns && !aligned(waited_ns, 8)))
        return KVQ8_ERR_INVALID_ARG;
    if (timeout_ns < 1000ull || timeout_ns > 10000000000ull) return KVQ8_ERR_INVALID_ARG;
    if (launch_bounded_wait_selftest(dev_status, timeout_ns, waited_ns, (cudaStream_t)stream) != cudaSuccess)
        return KVQ8_ERR_CUDA;
    return KVQ8_OK;
}

size_t kvq4_code_pool_bytes(int num_blocks, int nkv, int hd, int block_size) {
    if (num_blocks < 0 || nkv < 0 || hd < 0 || block_size < 0) return 0;
    return (size_t)num_blocks * nkv * block_size * (hd / 2);
}

size_t kvq4_param_pool_bytes(int num_blocks, int nkv, int block_size) {
    if (num_blocks < 0 || nkv < 0 || block_size < 0) return 0;
    return (size_t)num_blocks * nkv * block_size * 4 * sizeof(float);
}

size_t kvq4_cache_bytes_per_token(int nkv, int hd) {
    if (nkv < 0 || hd < 0) return 0;
    return (size_t)nkv * 2 * ((size_t)hd / 2 + 4 * sizeof(float));
}

kvq8_status kvq4_quantize_append(const float *k_new, const float *v_new, int batch, int n_new,
                                 int nkv, int hd, const int32_t *start_pos,
                                 const int32_t *block_table, int max_blocks, int block_size,
                                 int num_blocks, uint8_t *k_codes, uint8_t *v_codes,
                                 float *k_param, float *v_param, uint32_t *dev_status,
                                 void *stream) {
    kvq8_status st = check_shape(hd, block_size);
    if (st != KVQ8_OK) return st;
    if (batch < 0 || n_new < 0 || nkv <= 0 || num_blocks <= 0 || max_blocks <= 0)
        return KVQ8_ERR_INVALID_ARG;
    if (max_blocks > 2147483647 / kBS) return KVQ8_ERR_UNSUPPORTED;
    if (batch > kMaxGridYZ || nkv > kMaxGridYZ) return KVQ8_ERR_UNSUPPORTED;
    if (batch == 0 || n_new == 0) return KVQ8_OK;
    if (!k_new || !v_new || !start_pos || !block_table || !k_codes || !v_codes || !k_param ||
        !v_param)
        return KVQ8_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_codes, 16) ||
        !aligned(v_codes, 16) || !aligned(k_param, 16) || !aligned(v_param, 16) ||
        !aligned(start_pos, 4) || !aligned(block_table, 4))
        return KVQ8_ERR_INVALID_ARG;
    Int4AppendParams p;
    p.k_new = k_new;
    p.v_new = v_new;
    p.batch = batch;
    p.n_new = n_new;
    p.nkv = nkv;
    p.start_pos = start_pos;
    p.block_table = block_table;
    p.max_blocks = max_blocks;
    p.num_blocks = num_blocks;
    p.k_codes = k_codes;
    p.v_codes = v_codes;
    p.k_param = k_param;
    p.v_param = v_param;
    p.dev_status = dev_status;
    if (launch_int4_append(p, (cudaStream_t)stream) != cudaSuccess) return KVQ8_ERR_CUDA;
    return KVQ8_OK;
}

// The 4-bit decode, and with k_new / v_new a decode step (the split kernel
// also appends the new token at ctx_lens[b] - 1).
static kvq8_status run_kvq4_decode(const float *q, const float *k_new, const float *v_new, int batch, int nqh,
                                   int nkv, int hd, const uint8_t *k_codes, const uint8_t *v_codes,
                                   const float *k_param, const float *v_param, int num_blocks,
                                   const int32_t *block_table, int max_blocks, int block_size,
                                   const int32_t *ctx_lens, float sm_scale, float *out, void *workspace,
                                   size_t workspace_bytes, uint32_t *dev_status, void *stream) {
    kvq8_status st = check_decode_args(q, batch, nqh, nkv, hd, (const int8_t *)k_codes,
                                       (const int8_t *)v_codes, k_param, v_param, num_blocks,
                                       block_table, max_blocks, block_size, ctx_lens);
    if (st != KVQ8_OK || batch == 0) return st;
    if (!out || !aligned(out, 16) || !isfinite(sm_scale)) return KVQ8_ERR_INVALID_ARG;
    DecodeParams c;
    DecodePlan plan;
    st = fill_decode_params(q, batch, nqh, nkv, nullptr, nullptr, nullptr, nullptr, num_blocks,
                            block_table, max_blocks, ctx_lens, sm_scale, workspace,
                            workspace_bytes, dev_status, &c, &plan);
    if (st != KVQ8_OK) return st;
    c.out = out;
    Int4DecodeParams p;
    p.q = q;
    p.k_new = k_new;
    p.v_new = v_new;
    p.n4_blocks = nullptr;
    p.batch = batch;
    p.nqh = nqh;
    p.nkv = nkv;
    p.k_codes = k_codes;
    p.v_codes = v_codes;
    p.k_param = k_param;
    p.v_param = v_param;
    p.num_blocks = num_blocks;
    p.block_table = block_table;
    p.max_blocks = max_blocks;
    p.ctx_lens = ctx_lens;
    p.sm_scale_log2 = c.sm_scale_log2;
    if (!make_int4_plan(batch, nkv, max_blocks, int4_resident_ctas(plan.group), &p.nsplit,
                        &p.split_tokens))
        return KVQ8_ERR_INVALID_ARG;
    p.ws_meta = c.ws_meta;
    p.ws_ml = c.ws_ml;
    p.ws_acc = c.ws_acc;
    p.dev_status = dev_status;
    cudaStream_t s = (cudaStream_t)stream;
    if (launch_int4_decode_split(p, plan.group, s) != cudaSuccess) return KVQ8_ERR_CUDA;
    // the split's records sit at u * nsplit + j: a merge without the directory
    // when they fit its registers
    const cudaError_t e = p.nsplit <= 8 ? launch_decode_combine_fixed(c, plan.group, p.nsplit, s)
                                        : launch_decode_combine(c, plan.group, s);
    if (e != cudaSuccess) return KVQ8_ERR_CUDA;
    return KVQ8_OK;
}

kvq8_status kvq4_decode_attn(const float *q, int batch, int nqh, int nkv, int hd,
                             const uint8_t *k_codes, const uint8_t *v_codes, const float *k_param,
                             const float *v_param, int num_blocks, const int32_t *block_table,
                             int max_blocks, int block_size, const int32_t *ctx_lens,
                             float sm_scale, float *out, void *workspace, size_t workspace_bytes,
                             uint32_t *dev_status, void *stream) {
    return run_kvq4_decode(q, nullptr, nullptr, batch, nqh, nkv, hd, k_codes, v_codes, k_param, v_param,
                           num_blocks, block_table, max_blocks, block_size, ctx_lens, sm_scale, out, workspace,
                           workspace_bytes, dev_status, stream);
}

kvq8_status kvq4_decode_step(const float *q, const float *k_new, const float *v_new, int batch, int nqh,
                             int nkv, int hd, uint8_t *k_codes, uint8_t *v_codes, float *k_param,
                             float *v_param, int num_blocks, const int32_t *block_table, int max_blocks,
                             int block_size, const int32_t *ctx_lens, float sm_scale, float *out,
                             void *workspace, size_t workspace_bytes, uint32_t *dev_status, void *stream) {
    if (batch > 0 && (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16)))
        return KVQ8_ERR_INVALID_ARG;
    return run_kvq4_decode(q, k_new, v_new, batch, nqh, nkv, hd, k_codes, v_codes, k_param, v_param,
                           num_blocks, block_table, max_blocks, block_size, ctx_lens, sm_scale, out, workspace,
                           workspace_bytes, dev_status, stream);
}

size_t kvf32_pool_bytes(int num_blocks, int nkv, int hd, int block_size) {
    if (num_blocks < 0 || nkv < 0 || hd < 0 || block_size < 0) return 0;
    return (size_t)num_blocks * nkv * block_size * hd * sizeof(float);
}

size_t kvf32_cache_bytes_per_token(int nkv, int hd) {
    if (nkv < 0 || hd < 0) return 0;
    return (size_t)nkv * 2 * (size_t)hd * sizeof(float);
}

kvq8_status kvf32_append(const float *k_new, const float *v_new, int batch, int n_new, int nkv,
                         int hd, const int32_t *start_pos, const int32_t *block_table,
                         int max_blocks, int block_size, int num_blocks, float *k_cache,
                         float *v_cache, uint32_t *dev_status, void *stream) {
    kvq8_status st = check_shape(hd, block_size);
    if (st != KVQ8_OK) return st;
    if (batch < 0 || n_new < 0 || nkv <= 0 || num_blocks <= 0 || max_blocks <= 0)
        return KVQ8_ERR_INVALID_ARG;
    if (max_blocks > 2147483647 / kBS) return KVQ8_ERR_UNSUPPORTED;
    if (batch > kMaxGridYZ || nkv > kMaxGridYZ) return KVQ8_ERR_UNSUPPORTED;
    if (batch == 0 || n_new == 0) return KVQ8_OK;
    if (!k_new || !v_new || !start_pos || !block_table || !k_cache || !v_cache)
        return KVQ8_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(start_pos, 4) || !aligned(block_table, 4))
        return KVQ8_ERR_INVALID_ARG;
    F32AppendParams p;
    p.k_new = k_new;
    p.v_new = v_new;
    p.batch = batch;
    p.n_new = n_new;
    p.nkv = nkv;
    p.start_pos = start_pos;
    p.block_table = block_table;
    p.max_blocks = max_blocks;
    p.num_blocks = num_blocks;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.dev_status = dev_status;
    if (launch_f32_append(p, (cudaStream_t)stream) != cudaSuccess) return KVQ8_ERR_CUDA;
    return KVQ8_OK;
}

kvq8_status kvf32_decode_attn(const float *q, int batch, int nqh, int nkv, int hd,
                              const float *k_cache, const float *v_cache, int num_blocks,
                              const int32_t *block_table, int max_blocks, int block_size,
                              const int32_t *ctx_lens, float sm_scale, float *out,
                              void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                              void *stream) {
    // the scale arguments of the shared check are the caches themselves (non-null, aligned)
    kvq8_status st = check_decode_args(q, batch, nqh, nkv, hd, (const int8_t *)k_cache,
                                       (const int8_t *)v_cache, k_cache, v_cache, num_blocks,
                                       block_table, max_blocks, block_size, ctx_lens);
    if (st != KVQ8_OK || batch == 0) return st;
    if (!out || !aligned(out, 16) || !isfinite(sm_scale)) return KVQ8_ERR_INVALID_ARG;
    DecodeParams c;
    DecodePlan plan;
    st = fill_decode_params(q, batch, nqh, nkv, nullptr, nullptr, nullptr, nullptr, num_blocks,
                            block_table, max_blocks, ctx_lens, sm_scale, workspace,
                            workspace_bytes, dev_status, &c, &plan);
    if (st != KVQ8_OK) return st;
    c.out = out;
    F32DecodeParams p;
    p.q = q;
    p.batch = batch;
    p.nqh = nqh;
    p.nkv = nkv;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.num_blocks = num_blocks;
    p.block_table = block_table;
    p.max_blocks = max_blocks;
    p.ctx_lens = ctx_lens;
    p.sm_scale_log2 = c.sm_scale_log2;
    if (!make_f32_plan(batch, nkv, max_blocks, &p.nsplit, &p.split_tokens))
        return KVQ8_ERR_INVALID_ARG;
    p.ws_meta = c.ws_meta;
    p.ws_ml = c.ws_ml;
    p.ws_acc = c.ws_acc;
    p.dev_status = dev_status;
    cudaStream_t s = (cudaStream_t)stream;
    if (launch_f32_decode_split(p, plan.group, s) != cudaSuccess) return KVQ8_ERR_CUDA;
    if (launch_decode_combine(c, plan.group, s) != cudaSuccess) return KVQ8_ERR_CUDA;
    return KVQ8_OK;
}

size_t kvmix_decode_workspace_bytes(int batch, int nqh, int nkv, int hd, int max_blocks,
                                    int block_size) {
    const size_t one = kvq8_decode_workspace_bytes(batch, nqh, nkv, hd, max_blocks, block_size);
    return 2 * one;
}

kvq8_status kvmix_requantize(int batch, int nkv, int hd, const int8_t *k_pool, const int8_t *v_pool,
                             const float *k_scale, const float *v_scale, int num_blocks8,
                             const int32_t *table8, uint8_t *k_codes, uint8_t *v_codes,
                             float *k_param, float *v_param, int num_blocks4, const int32_t *table4,
                             int max_blocks, int block_size, const int32_t *blk_from,
                             const int32_t *blk_to, int max_count, uint32_t *dev_status,
                             void *stream) {
    kvq8_status st = check_shape(hd, block_size);
    if (st != KVQ8_OK) return st;
    if (batch < 0 || nkv <= 0 || num_blocks8 <= 0 || num_blocks4 <= 0 || max_blocks <= 0 ||
        max_count < 0)
        return KVQ8_ERR_INVALID_ARG;
    if (max_blocks > 2147483647 / kBS) return KVQ8_ERR_UNSUPPORTED;
    if (batch > kMaxGridYZ || nkv > kMaxGridYZ) return KVQ8_ERR_UNSUPPORTED;
    if (batch == 0 || max_count == 0) return KVQ8_OK;
    if (!k_pool || !v_pool || !k_scale || !v_scale || !table8 || !k_codes || !v_codes ||
        !k_param || !v_param || !table4 || !blk_from || !blk_to)
        return KVQ8_ERR_INVALID_ARG;
    if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(k_scale, 4) ||
        !aligned(v_scale, 4) || !aligned(k_codes, 16) || !aligned(v_codes, 16) ||
        !aligned(k_param, 16) || !aligned(v_param, 16) || !aligned(table8, 4) ||
        !aligned(table4, 4) || !aligned(blk_from, 4) || !aligned(blk_to, 4))
        return KVQ8_ERR_INVALID_ARG;
    Int4RequantParams p;
    p.batch = batch;
    p.nkv = nkv;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.num_blocks8 = num_blocks8;
    p.table8 = table8;
    p.k_codes = k_codes;
    p.v_codes = v_codes;
    p.k_param = k_param;
    p.v_param = v_param;
    p.num_blocks4 = num_blocks4;
    p.table4 = table4;
    p.max_blocks = max_blocks;
    p.blk_from = blk_from;
    p.blk_to = blk_to;
    p.max_count = max_count;
    p.dev_status = dev_status;
    if (launch_int4_requantize(p, (cudaStream_t)stream) != cudaSuccess) return KVQ8_ERR_CUDA;
    return KVQ8_OK;
}

kvq8_status kvmix_decode_attn(const float *q, int batch, int nqh, int nkv, int hd,
                              const int8_t *k_pool, const int8_t *v_pool, const float *k_scale,
                              const float *v_scale, int num_blocks8, const int32_t *table8,
                              const uint8_t *k_codes, const uint8_t *v_codes, const float *k_param,
                              const float *v_param, int num_blocks4, const int32_t *table4,
                              int max_blocks, int block_size, const int32_t *ctx_lens,
                              const int32_t *n4_blocks, float sm_scale, float *out, void *workspace,
                              size_t workspace_bytes, uint32_t *dev_status, void *stream) {
    kvq8_status st = check_decode_args(q, batch, nqh, nkv, hd, k_pool, v_pool, k_scale, v_scale,
                                       num_blocks8, table8, max_blocks, block_size, ctx_lens);
    if (st != KVQ8_OK || batch == 0) return st;
    st = check_decode_args(q, batch, nqh, nkv, hd, (const int8_t *)k_codes, (const int8_t *)v_codes,
                           k_param, v_param, num_blocks4, table4, max_blocks, block_size, ctx_lens);
    if (st != KVQ8_OK) return st;
    if (!out || !aligned(out, 16) || !isfinite(sm_scale) || !n4_blocks || !aligned(n4_blocks, 4))
        return KVQ8_ERR_INVALID_ARG;
    DecodePlan plan;
    if (!make_decode_plan(batch, nqh, nkv, max_blocks, &plan)) return KVQ8_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < 2 * plan.bytes)
        return KVQ8_ERR_WORKSPACE;
    // first half: the int8 split's records; second half: the 4-bit split's
    DecodeParams c, c4;
    st = fill_decode_params(q, batch, nqh, nkv, k_pool, v_pool, k_scale, v_scale, num_blocks8,
                            table8, max_blocks, ctx_lens, sm_scale, workspace, plan.bytes,
                            dev_status, &c, &plan);
    if (st != KVQ8_OK) return st;
    st = fill_decode_params(q, batch, nqh, nkv, nullptr, nullptr, nullptr, nullptr, num_blocks4,
                            table4, max_blocks, ctx_lens, sm_scale, (char *)workspace + plan.bytes,
                            plan.bytes, dev_status, &c4, &plan);
    if (st != KVQ8_OK) return st;
    c.out = out;
    c.first_q8_block = n4_blocks;
    c.ws_meta2 = c4.ws_meta;
    c.ws_ml2 = c4.ws_ml;
    c.ws_acc2 = c4.ws_acc;
    Int4DecodeParams p;
    p.q = q;
    p.k_new = nullptr;
    p.v_new = nullptr;
    p.n4_blocks = n4_blocks;
    p.batch = batch;
    p.nqh = nqh;
    p.nkv = nkv;
    p.k_codes = k_codes;
    p.v_codes = v_codes;
    p.k_param = k_param;
    p.v_param = v_param;
    p.num_blocks = num_blocks4;
    p.block_table = table4;
    p.max_blocks = max_blocks;
    p.ctx_lens = ctx_lens;
    p.sm_scale_log2 = c.sm_scale_log2;
    if (!make_int4_plan(batch, nkv, max_blocks, int4_resident_ctas(plan.group), &p.nsplit,
                        &p.split_tokens))
        return KVQ8_ERR_INVALID_ARG;
    p.ws_meta = c4.ws_meta;
    p.ws_ml = c4.ws_ml;
    p.ws_acc = c4.ws_acc;
    p.dev_status = dev_status;
    cudaStream_t s = (cudaStream_t)stream;
    if (launch_int4_decode_split(p, plan.group, s) != cudaSuccess) return KVQ8_ERR_CUDA;
    if (launch_decode_split(c, plan.group, s) != cudaSuccess) return KVQ8_ERR_CUDA;
    if (launch_decode_combine(c, plan.group, s) != cudaSuccess) return KVQ8_ERR_CUDA;
    return KVQ8_OK;
}

}  // extern "C"
