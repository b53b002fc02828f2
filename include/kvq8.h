/*
 * kvq8.h -- C ABI of libkvq8: decode attention over a paged INT8 KV cache on
 * NVIDIA GB300 (sm_103a).
 *
 * The method (pages of the "0.8MB 跑通 Qwen" tutorial series):
 *   [Day 9-1] "推理引擎的 KV 也量化——q8 KV 把缓存与 decode 带宽压到一半", §2:
 *             K/V stored as int8 with one fp32 scale per (token, kv head).
 *   [Day 9-2] "flash_attn_single_q_q8_neon——单 q 单遍扫全 KV", §1-§3: the query
 *             quantised once in 32-element blocks, int8 dot products per block,
 *             scales applied afterwards, online softmax, one divide at the end.
 *   [Day 9-3] "q8 KV 精度对照——量化进注意力，输出差多少", §2: the quantisation rule
 *             scale = max_abs/127, code = round(v/scale) clamped to [-127, 127].
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument is a DEVICE pointer owned by the caller, except
 *   `stream` (a cudaStream_t, NULL = legacy default stream).  The library
 *   allocates no memory, never synchronises the device or the stream, and
 *   keeps no state between calls apart from a per-device cache of device
 *   attributes.  A device pointer may also be the device address of
 *   page-locked host memory mapped into the device's address space
 *   (kvq8_host_device_pointer): the kernels then read or write that host
 *   memory themselves over the host link, which pays for the small per-step
 *   buffers (q, the new token's k_new and v_new, out), not for the pools or
 *   the workspace.
 * - The last kernel of every decode call (the split merge) lets the next
 *   kernel of the stream launch before it completes (programmatic dependent
 *   launch): a kernel launched after it with the programmatic stream
 *   serialisation attribute must wait for it (griddepcontrol.wait /
 *   cudaGridDependencySynchronize) before reading `out`; every kernel of this
 *   library does.  Kernels launched without that attribute start after it
 *   completes, as usual.
 * - Work is enqueued asynchronously on `stream`.  Argument errors are
 *   detected on the host and returned before anything is enqueued.  A
 *   failed launch returns KVQ8_ERR_CUDA (the CUDA error is left for
 *   cudaGetLastError()).  Faults the kernels detect at run time (a block id
 *   outside the pool, a context length beyond the block table) are OR-ed as
 *   KVQ8_DEV_* bits into *dev_status when dev_status is non-NULL; the
 *   offending tokens are skipped, never read or written out of bounds.
 * - Rounding: every float->int step rounds half to even in IEEE fp32, and
 *   every fp32 division is IEEE-correct, so quantised codes and scales are
 *   reproducible bit for bit on any IEEE machine.
 * - Non-finite inputs (the pages state the rules for finite values only): a
 *   unit of quantisation -- a K/V row of the int8 cache, a 64-value group of
 *   the 4-bit cache, a 32-value block of the query in the int8 decode --
 *   that holds a NaN or an infinity is quantised as if all its values were
 *   zero, and KVQ8_DEV_NONFINITE is set.  So an int8 row gets scale 0 and
 *   codes 0, a 4-bit group scale 1, zero -0 and codes 0, a query block scale
 *   1/127 and codes 0; the cache and the outputs stay finite.  The fp32-query
 *   decodes (4-bit and fp32 caches) and the fp32 cache take their inputs as
 *   they are: IEEE arithmetic, unflagged.
 * - Supported shapes: hd == 128, block_size == 256, nqh % nkv == 0 with
 *   G = nqh/nkv in {1, 2, 4, 8}.  Anything else returns KVQ8_ERR_UNSUPPORTED.
 *
 * Cache layout (pool of num_blocks physical blocks, shared by all sequences)
 * --------------------------------------------------------------------------
 * A (block, kv head) tile holds block_size = 256 tokens:
 *   k_pool  int8  [num_blocks][nkv][256][128]      token-major rows; the 16-byte
 *                 chunk j (dims 16j..16j+15) of the row of slot t is stored at
 *                 chunk position j ^ (t & 7)
 *   v_pool  int8  [num_blocks][nkv][4][128][64]    per 64-token quarter, dim-major:
 *                 the code of slot t, dim d is at [t / 64][d][t % 64]
 *   k_scale fp32  [num_blocks][nkv][256]           one scale per (token, head)
 *   v_scale fp32  [num_blocks][nkv][256]
 * This is the order in which the decode kernel consumes the cache: every
 * 64-token window is four contiguous runs (8 KiB of K, 8 KiB of V, 256 B of
 * each scale) that one bulk copy each brings into shared memory, where the
 * chunk permutation keeps the reads free of bank conflicts.
 *   block_table int32 [batch][max_blocks]: logical block j of sequence b lives
 *   in physical block block_table[b*max_blocks + j]; token t of sequence b is
 *   slot t % block_size of logical block t / block_size.
 * The pointers must be 16-byte aligned.  One tile of K or V is 32 KiB
 * contiguous; a token costs 2*hd + 8 bytes per kv head (2112 bytes per token
 * for nkv = 8).
 */
#ifndef KVQ8_H
#define KVQ8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvq8_status {
    KVQ8_OK = 0,
    KVQ8_ERR_INVALID_ARG = 1,  /* NULL pointer, negative or inconsistent size, misalignment */
    KVQ8_ERR_UNSUPPORTED = 2,  /* shape outside the supported set above */
    KVQ8_ERR_WORKSPACE = 3,    /* workspace NULL, not 256-byte aligned, or too small */
    KVQ8_ERR_CUDA = 4          /* a CUDA runtime call or kernel launch failed */
} kvq8_status;

/* Bits the kernels OR into *dev_status. */
#define KVQ8_DEV_BAD_BLOCK_ID 0x1u   /* a needed block-table entry is outside [0, num_blocks) */
#define KVQ8_DEV_BAD_CTX_LEN 0x2u    /* ctx_lens[b] < 0 or > max_blocks * block_size */
#define KVQ8_DEV_BAD_POSITION 0x4u   /* append position start_pos[b]+i outside the block table */
#define KVQ8_DEV_TIMEOUT 0x8u        /* an internal pipeline wait gave up (never expected); the
                                        affected results are unspecified */
#define KVQ8_DEV_NONFINITE 0x10u     /* a K/V row, a 4-bit group or a query 32-block held a NaN
                                        or an infinity and was quantised as zeros (see below) */

#define KVQ8_HEAD_DIM 128
#define KVQ8_BLOCK_SIZE 256
#define KVQ8_Q_BLOCK 32

/* Human-readable name of a status code (static string, never NULL). */
const char *kvq8_status_str(int status);

/* ABI revision of this header; bumped on any incompatible change. */
int kvq8_abi_version(void);

/* ---------------------------------------------------------------- sizes --- */

/* Bytes of one int8 pool (k_pool or v_pool) and of one scale array. */
size_t kvq8_kv_pool_bytes(int num_blocks, int nkv, int hd, int block_size);
size_t kvq8_scale_pool_bytes(int num_blocks, int nkv, int block_size);

/* Cache bytes one token occupies in one layer: int8 K and V rows plus one
 * fp32 scale each, for every kv head ([Day 9-1] §2: 2112 for nkv=8, hd=128). */
size_t kvq8_cache_bytes_per_token(int nkv, int hd);

/* ------------------------------------------------------- quantize-append --- */

/*
 * kvq8_quantize_append -- quantise new K/V rows and write them into the cache.
 * [Day 9-3] §2 / [Day 9-1] §2 (kv_quantize_per_head): for each (token, kv head)
 * row of hd values, scale = max|v| / 127 (fp32), code = round_half_even(v /
 * scale) clamped to [-127, 127]; an all-zero row gets scale 0 and codes 0.
 *
 *   k_new, v_new  fp32 [batch][n_new][nkv][hd]: the rows to append
 *   start_pos     int32 [batch]: position of the first new token of each
 *                 sequence; token i goes to position start_pos[b] + i
 *   block_table   int32 [batch][max_blocks] (see layout above)
 *   num_blocks    physical blocks in the pool (bounds for block ids)
 *   k_pool, v_pool, k_scale, v_scale   the cache, written in place
 *   dev_status    optional uint32 word receiving KVQ8_DEV_* bits
 * Rows whose position is negative or beyond max_blocks*block_size, or whose
 * block id is out of range, are skipped and flagged.  batch == 0 or
 * n_new == 0 is a no-op.
 */
kvq8_status kvq8_quantize_append(const float *k_new, const float *v_new,
                                 int batch, int n_new, int nkv, int hd,
                                 const int32_t *start_pos,
                                 const int32_t *block_table, int max_blocks,
                                 int block_size, int num_blocks,
                                 int8_t *k_pool, int8_t *v_pool,
                                 float *k_scale, float *v_scale,
                                 uint32_t *dev_status, void *stream);

/*
 * kvq8_quantize_append_host -- kvq8_quantize_append with the new rows in host
 * memory: k_new_host and v_new_host (fp32 [batch][n_new][nkv][hd]) are copied
 * into the caller's device buffers k_new and v_new of the same size (one
 * cudaMemcpyAsync each, on `stream`), then appended.  Asynchronous like every
 * call here: the host buffers must not change until the stream has passed
 * this point; page-locked host memory lets the copies run at full speed.
 * Returns as kvq8_quantize_append (all arguments are checked before anything
 * is queued); KVQ8_ERR_INVALID_ARG also for a null host pointer when there is
 * something to append; KVQ8_ERR_CUDA when a copy cannot be queued.
 */
kvq8_status kvq8_quantize_append_host(const float *k_new_host, const float *v_new_host,
                                      float *k_new, float *v_new,
                                      int batch, int n_new, int nkv, int hd,
                                      const int32_t *start_pos,
                                      const int32_t *block_table, int max_blocks,
                                      int block_size, int num_blocks,
                                      int8_t *k_pool, int8_t *v_pool,
                                      float *k_scale, float *v_scale,
                                      uint32_t *dev_status, void *stream);

/* ------------------------------------------------------- query quantize --- */

/*
 * kvq8_quantize_q -- 32-block query quantisation, exposed on its own so that
 * the step the decode performs in its prologue can be checked bit for bit.
 * [Day 9-2] §2 segment 1: per 32-element block qm = max|x| (qm = 1 when
 * qm < 1e-6), block scale = qm * (1/127), code = round_half_even(x * (127/qm))
 * clamped to [-128, 127].  A block holding a NaN or an infinity is quantised
 * as zeros, as in the decode; this call has no status word to flag it in.
 *
 *   q         fp32 [n_rows][hd]
 *   q_codes   int8 [n_rows][hd]
 *   q_scales  fp32 [n_rows][hd/32]
 */
kvq8_status kvq8_quantize_q(const float *q, int64_t n_rows, int hd,
                            int8_t *q_codes, float *q_scales, void *stream);

/* --------------------------------------------------------------- decode --- */

/*
 * kvq8_decode_workspace_bytes -- bytes of device workspace kvq8_decode_split /
 * kvq8_decode_attn need for these sizes (the split-KV partial results).  Pure
 * host arithmetic; returns 0 for unsupported or invalid sizes.
 */
size_t kvq8_decode_workspace_bytes(int batch, int nqh, int nkv, int hd,
                                   int max_blocks, int block_size);

/*
 * kvq8_decode_attn -- single-query decode attention over the int8 cache,
 * [Day 9-2] §1-§3, split over the context and merged:
 *   per kv head, the G = nqh/nkv query heads j with j / G == kv head are
 *   quantised in 32-blocks (as kvq8_quantize_q); for every cached token t,
 *   s_t = (sum_b dot32_b(q_codes, k_codes_t) * q_scale_b) * k_scale_t * sm_scale
 *   with exact int32 block dots; softmax over t with a running maximum, V
 *   accumulated as int8 code * (weight * v_scale_t) in fp32; one division by
 *   the softmax sum at the end.  Sequences with ctx_lens[b] == 0 yield 0.
 *
 *   q             fp32 [batch][nqh][hd]: one query token per sequence
 *   ctx_lens      int32 [batch]: tokens 0 .. ctx_lens[b]-1 are attended
 *   sm_scale      softmax scale, normally 1/sqrt(hd)
 *   out           fp32 [batch][nqh][hd]
 *   workspace     at least kvq8_decode_workspace_bytes(...) bytes, 256-byte
 *                 aligned; its contents need no initialisation and are
 *                 overwritten; calls that share it must not overlap in time
 * Decode layers of one model step can be folded into `batch` (one row of q,
 * block_table and ctx_lens per (layer, sequence), all in one shared pool).
 */
kvq8_status kvq8_decode_attn(const float *q, int batch, int nqh, int nkv, int hd,
                             const int8_t *k_pool, const int8_t *v_pool,
                             const float *k_scale, const float *v_scale,
                             int num_blocks, const int32_t *block_table,
                             int max_blocks, int block_size,
                             const int32_t *ctx_lens, float sm_scale,
                             float *out, void *workspace, size_t workspace_bytes,
                             uint32_t *dev_status, void *stream);

/*
 * kvq8_decode_split / kvq8_decode_combine -- the two launches kvq8_decode_attn
 * makes, exposed separately so that each can be timed on its own.  split
 * writes per-split partial results (running max, softmax sum, unnormalised V
 * accumulator) into the workspace; combine merges them per query head:
 * M = max_i M_i, S = sum_i S_i e^(M_i - M), out = sum_i acc_i e^(M_i - M) / S.
 * They must be called with the same sizes and workspace, split first.
 */
kvq8_status kvq8_decode_split(const float *q, int batch, int nqh, int nkv, int hd,
                              const int8_t *k_pool, const int8_t *v_pool,
                              const float *k_scale, const float *v_scale,
                              int num_blocks, const int32_t *block_table,
                              int max_blocks, int block_size,
                              const int32_t *ctx_lens, float sm_scale,
                              void *workspace, size_t workspace_bytes,
                              uint32_t *dev_status, void *stream);

kvq8_status kvq8_decode_combine(int batch, int nqh, int nkv, int hd,
                                int max_blocks, int block_size,
                                const int32_t *ctx_lens,
                                const void *workspace, size_t workspace_bytes,
                                float *out, void *stream);

/*
 * kvq8_decode_step -- one decode step in one call: append the step's new
 * token of every sequence at position ctx_lens[b] - 1 and attend over the
 * context including it.  Same results as kvq8_quantize_append (n_new = 1,
 * start_pos[b] = ctx_lens[b] - 1) followed by kvq8_decode_attn, in two
 * launches: the split kernel also appends the new token (the CTA that decodes
 * a unit's last 64-token stage quantises the token into that stage and into
 * the pools), then the merge.  Both are programmatic dependents of the kernel
 * before them in the stream, so that their launches overlap it; each waits
 * for that kernel's results before it reads anything.  The block holding a
 * sequence's new position must belong to that sequence alone (no other
 * sequence of the call may read it in the same call).
 *
 *   k_new, v_new  fp32 [batch][nkv][hd]: the step's token ([Day 9-3] §2 rule)
 *                 (sequences with ctx_lens[b] == 0 append nothing and yield 0;
 *                 a ctx_lens[b] beyond the table is flagged, clamped, and
 *                 appends nothing)
 *   pools         written at the new token's slot only
 * Other arguments, workspace included, as kvq8_decode_attn.
 */
kvq8_status kvq8_decode_step(const float *q, const float *k_new, const float *v_new,
                             int batch, int nqh, int nkv, int hd,
                             int8_t *k_pool, int8_t *v_pool, float *k_scale, float *v_scale,
                             int num_blocks, const int32_t *block_table,
                             int max_blocks, int block_size,
                             const int32_t *ctx_lens, float sm_scale, float *out,
                             void *workspace, size_t workspace_bytes,
                             uint32_t *dev_status, void *stream);

/*
 * kvq8_decode_step_ex -- kvq8_decode_step with flags (0 = kvq8_decode_step).
 *
 * KVQ8_STEP_CACHE_READY: the caller vouches that the cache blocks this call
 * reads (apart from its new tokens' slots, which it writes itself),
 * block_table and ctx_lens held their final values before the kernel that
 * precedes this call in the stream began (they are not written by that
 * kernel, nor by anything it does not wait for).  The split kernel then runs
 * its prologue and starts copying the cache into shared memory without
 * waiting for that kernel; only the reads of q, k_new and v_new and the
 * writes of the workspace, the pools' new-token slots and out wait for it.
 * A decode that runs one layer per call after the layer's own projections
 * (which write q, k_new and v_new only) meets this; so does a chain of steps
 * that differ only in those inputs.  Results are identical with and without
 * the flag.
 * Flags outside KVQ8_STEP_CACHE_READY return KVQ8_ERR_INVALID_ARG.
 */
#define KVQ8_STEP_CACHE_READY 0x1u
kvq8_status kvq8_decode_step_ex(const float *q, const float *k_new, const float *v_new,
                                int batch, int nqh, int nkv, int hd,
                                int8_t *k_pool, int8_t *v_pool, float *k_scale, float *v_scale,
                                int num_blocks, const int32_t *block_table,
                                int max_blocks, int block_size,
                                const int32_t *ctx_lens, float sm_scale, float *out,
                                void *workspace, size_t workspace_bytes,
                                uint32_t *dev_status, uint32_t flags, void *stream);

/*
 * kvq8_decode_step_host -- kvq8_decode_step from host memory and back, the
 * call a serving loop makes each step: the inputs q_host (fp32
 * [batch][nqh][hd]), k_new_host and v_new_host (fp32 [batch][nkv][hd]) and the
 * result out_host ([batch][nqh][hd]) are in host memory.  When all four are
 * page-locked and mapped into the device's address space (every page-locked
 * allocation, on a system with unified addressing) and 16-byte aligned, the
 * kernels read the inputs from host memory and write the result there
 * themselves: nothing is copied and the device buffers q, k_new, v_new and
 * out are left untouched.  Otherwise the inputs are copied into the caller's
 * device buffers q, k_new and v_new, the step runs, and its result is copied
 * from the device buffer out into out_host (one cudaMemcpyAsync per copy).
 * Everything is queued on `stream`; the caller synchronises the stream before
 * reading out_host, and the input host buffers must not change until then.
 * Returns as kvq8_decode_step (all arguments, the device buffers included, are
 * checked before anything is queued); KVQ8_ERR_INVALID_ARG also for a null
 * host pointer when batch > 0; KVQ8_ERR_CUDA when a copy cannot be queued.
 */
kvq8_status kvq8_decode_step_host(const float *q_host, const float *k_new_host,
                                  const float *v_new_host, float *out_host,
                                  float *q, float *k_new, float *v_new,
                                  int batch, int nqh, int nkv, int hd,
                                  int8_t *k_pool, int8_t *v_pool,
                                  float *k_scale, float *v_scale,
                                  int num_blocks, const int32_t *block_table,
                                  int max_blocks, int block_size,
                                  const int32_t *ctx_lens, float sm_scale,
                                  float *out, void *workspace, size_t workspace_bytes,
                                  uint32_t *dev_status, void *stream);

/*
 * kvq8_host_device_pointer -- not part of the pages' method: the device
 * address of host memory that the current device can access directly
 * (page-locked memory mapped into its address space; with unified addressing
 * every page-locked allocation is), provided it is 16-byte aligned there;
 * NULL for pageable, device, unknown or misaligned memory.  The result can be
 * passed wherever a call takes q, k_new, v_new or out.  Looked up once for
 * buffers that are reused every step, it saves kvq8_decode_step_host's
 * per-call lookup.
 */
const void *kvq8_host_device_pointer(const void *host_ptr);

/*
 * kvq8_selftest_bounded_wait -- not part of the pages' method: a check that
 * the kernels' bounded waits end.  Every wait of the decode kernels on a copy
 * or a shared-memory slot gives up after a bound, ORs KVQ8_DEV_TIMEOUT into
 * *dev_status and unwinds rather than spin forever.  This call launches one
 * warp that runs the same wait routine on an mbarrier phase that nothing
 * completes, bounded by timeout_ns (1 us .. 10 s), so the bound passes on
 * purpose: the warp then ORs KVQ8_DEV_TIMEOUT into *dev_status, writes the
 * nanoseconds it waited to *waited_ns (when non-NULL) and exits, leaving the
 * context usable.  dev_status (4-byte aligned) and waited_ns (8-byte aligned)
 * are device pointers; enqueued on `stream`.  KVQ8_ERR_INVALID_ARG for a NULL
 * or misaligned status word or a bound outside the range.
 */
kvq8_status kvq8_selftest_bounded_wait(uint32_t *dev_status, uint64_t timeout_ns,
                                       unsigned long long *waited_ns, void *stream);

/* -------------------------------------------- 4-bit cache (NEXT row) --- */

/*
 * The asymmetric INT4 group-64 cache of [UltraQuant] §3.2 ("方差均衡化分组量化的
 * 具体实现", its code): per group of 64 consecutive values of a (token, kv head)
 * row, scale = (max - min)/15 (1 when max == min), zero = round_half_even
 * (-min/scale) kept in fp32 (not clamped), code = clamp(round_half_even(x/scale
 * + zero), 0, 15), two codes per byte with the even element in the high
 * nibble; value = (code - zero) * scale.  The page's variance-dependent scale
 * tweak is marked there as an example, not the formula, and is not applied.
 *
 * Layout per (block, kv head) tile of 256 tokens (every code byte is the
 * page's pair: byte i of a row = code[2i] << 4 | code[2i+1]):
 *   k_codes uint8 [num_blocks][nkv][256][hd/2]       token-major rows
 *   v_codes uint8 [num_blocks][nkv][8][hd/2][32]     per 32-token chunk, byte
 *           column c (dims 2c, 2c+1) of its 32 tokens: token t of the chunk
 *           (r = t % 16) at position 4*(2*((r%8)/2) + t/16) + 2*(r%2) + r/8,
 *           the order in which the decode's tensor-core fragments take them
 *   k_param, v_param fp32  [num_blocks][nkv][256][4]  (scale0, zero0, scale1, zero1)
 * 160 bytes per (token, kv head): 1280 bytes per token per layer for nkv = 8.
 */
size_t kvq4_code_pool_bytes(int num_blocks, int nkv, int hd, int block_size);
size_t kvq4_param_pool_bytes(int num_blocks, int nkv, int block_size);
size_t kvq4_cache_bytes_per_token(int nkv, int hd);

/* kvq4_quantize_append -- as kvq8_quantize_append, into the 4-bit cache. */
kvq8_status kvq4_quantize_append(const float *k_new, const float *v_new,
                                 int batch, int n_new, int nkv, int hd,
                                 const int32_t *start_pos,
                                 const int32_t *block_table, int max_blocks,
                                 int block_size, int num_blocks,
                                 uint8_t *k_codes, uint8_t *v_codes,
                                 float *k_param, float *v_param,
                                 uint32_t *dev_status, void *stream);

/*
 * kvq4_decode_attn -- decode attention of the fp32 query over the dequantised
 * 4-bit cache ([UltraQuant] §4.1 / §5.3: dequantise, then standard attention):
 * s_t = sm_scale * q . dequant(k_t), softmax with a running maximum, fp32
 * accumulation of dequant(v_t), split over the context and merged as in
 * kvq8_decode_attn.  Workspace: kvq8_decode_workspace_bytes(...) for the same
 * sizes.  Other arguments as kvq8_decode_attn.
 */
kvq8_status kvq4_decode_attn(const float *q, int batch, int nqh, int nkv, int hd,
                             const uint8_t *k_codes, const uint8_t *v_codes,
                             const float *k_param, const float *v_param,
                             int num_blocks, const int32_t *block_table,
                             int max_blocks, int block_size,
                             const int32_t *ctx_lens, float sm_scale,
                             float *out, void *workspace, size_t workspace_bytes,
                             uint32_t *dev_status, void *stream);

/*
 * kvq4_decode_step -- one decode step over the 4-bit cache in one call: append
 * the step's new token of every sequence at position ctx_lens[b] - 1 (the
 * group-64 rule of kvq4_quantize_append) and attend over the context including
 * it.  Same results as kvq4_quantize_append (n_new = 1, start_pos[b] =
 * ctx_lens[b] - 1) followed by kvq4_decode_attn, in two launches: the split
 * kernel also appends the new token (the warp that decodes the 32-token chunk
 * holding it quantises the token into that chunk and into the cache), then
 * the merge.  Both are programmatic dependents of the kernel before them in
 * the stream; each waits for that kernel's results before it reads anything.
 * The block holding a sequence's new position must belong to that sequence
 * alone.
 *
 *   k_new, v_new  fp32 [batch][nkv][hd], 16-byte aligned (sequences with
 *                 ctx_lens[b] == 0 append nothing and yield 0; a ctx_lens[b]
 *                 beyond the table is flagged, clamped, and appends nothing)
 *   k_codes .. v_param  written at the new token's slot only
 * Other arguments, workspace included, as kvq4_decode_attn.
 */
kvq8_status kvq4_decode_step(const float *q, const float *k_new, const float *v_new,
                             int batch, int nqh, int nkv, int hd,
                             uint8_t *k_codes, uint8_t *v_codes, float *k_param, float *v_param,
                             int num_blocks, const int32_t *block_table,
                             int max_blocks, int block_size,
                             const int32_t *ctx_lens, float sm_scale, float *out,
                             void *workspace, size_t workspace_bytes,
                             uint32_t *dev_status, void *stream);

/* ------------------------- mixed precision by token age (NEXT row) --- */

/*
 * [UltraQuant] §3.3 (time-adaptive quantisation, its practical note): tokens
 * in a time block share one precision; recent blocks stay 8-bit and, as the
 * sequence grows, the oldest blocks are requantised to 4-bit.  Here a time
 * block is a cache block of 256 tokens: for sequence b the logical blocks
 * [0, n4_blocks[b]) live in the 4-bit cache (tiles table4[b][j]) and the
 * later ones in the int8 cache (tiles table8[b][j]); both tables have
 * max_blocks columns and are indexed by the logical block.  The page's 2-bit
 * tier is not defined there and is not built.
 *
 * kvmix_requantize -- for every sequence b, requantise the logical blocks
 * [blk_from[b], blk_to[b]) (whole 256-token tiles, K and V) from the int8
 * tiles to the 4-bit tiles: value = code * scale (fp32), then the 4-bit group
 * rule of kvq4_quantize_append.  max_count >= max_b (blk_to[b] - blk_from[b])
 * sizes the grid.  A range outside [0, max_blocks) or longer than max_count
 * sets KVQ8_DEV_BAD_POSITION (the part inside is still done); a tile id
 * outside its pool sets KVQ8_DEV_BAD_BLOCK_ID and is skipped.  The int8 tiles
 * are left as they were.  Whole tiles are converted: slots past a sequence's
 * last token are converted from whatever they hold (never read as tokens), and
 * a non-finite leftover there sets KVQ8_DEV_NONFINITE like any other.
 */
kvq8_status kvmix_requantize(int batch, int nkv, int hd,
                             const int8_t *k_pool, const int8_t *v_pool,
                             const float *k_scale, const float *v_scale,
                             int num_blocks8, const int32_t *table8,
                             uint8_t *k_codes, uint8_t *v_codes,
                             float *k_param, float *v_param,
                             int num_blocks4, const int32_t *table4,
                             int max_blocks, int block_size,
                             const int32_t *blk_from, const int32_t *blk_to, int max_count,
                             uint32_t *dev_status, void *stream);

/* Workspace of kvmix_decode_attn: twice kvq8_decode_workspace_bytes. */
size_t kvmix_decode_workspace_bytes(int batch, int nqh, int nkv, int hd, int max_blocks,
                                    int block_size);

/*
 * kvmix_decode_attn -- decode attention of sequence b over its tokens
 * [0, 256 * n4_blocks[b]) in the 4-bit cache (fp32 query against the
 * dequantised rows, as kvq4_decode_attn) and [256 * n4_blocks[b], ctx_lens[b])
 * in the int8 cache (the q8 method of kvq8_decode_attn): both splits' partial
 * results are merged by one combine, so the softmax is taken over the whole
 * context.  n4_blocks: device int32 [batch] (values clamped to
 * [0, max_blocks]).  Other arguments as kvq8_decode_attn and kvq4_decode_attn.
 */
kvq8_status kvmix_decode_attn(const float *q, int batch, int nqh, int nkv, int hd,
                              const int8_t *k_pool, const int8_t *v_pool,
                              const float *k_scale, const float *v_scale,
                              int num_blocks8, const int32_t *table8,
                              const uint8_t *k_codes, const uint8_t *v_codes,
                              const float *k_param, const float *v_param,
                              int num_blocks4, const int32_t *table4,
                              int max_blocks, int block_size,
                              const int32_t *ctx_lens, const int32_t *n4_blocks,
                              float sm_scale, float *out,
                              void *workspace, size_t workspace_bytes,
                              uint32_t *dev_status, void *stream);

/* --------------------------------------- fp32 cache (comparator row) --- */

/*
 * The fp32 K/V cache that [Day 9-1] §2-§3 keeps beside the int8 cache for
 * debugging and comparison, and that [Day 9-3] §1 takes as the unquantised arm
 * of its fp32-KV vs q8-KV experiment ("change one variable": the same
 * attention over raw fp32 K/V).  Here it is paged with the same block table
 * conventions as the int8 cache:
 *   k_cache, v_cache fp32 [num_blocks][nkv][256][hd]   token-major rows
 * 1024 bytes per (token, kv head): 8192 bytes per token per layer for nkv = 8,
 * against 2112 for the int8 cache.
 */
size_t kvf32_pool_bytes(int num_blocks, int nkv, int hd, int block_size);
size_t kvf32_cache_bytes_per_token(int nkv, int hd);

/*
 * kvf32_append -- copy the new tokens' fp32 K/V rows into the fp32 cache at
 * positions start_pos[b] + i.  Arguments as kvq8_quantize_append; k_cache and
 * v_cache 16-byte aligned.  Positions beyond the table and block ids outside
 * [0, num_blocks) are flagged in *dev_status and skipped.
 */
kvq8_status kvf32_append(const float *k_new, const float *v_new,
                         int batch, int n_new, int nkv, int hd,
                         const int32_t *start_pos,
                         const int32_t *block_table, int max_blocks,
                         int block_size, int num_blocks,
                         float *k_cache, float *v_cache,
                         uint32_t *dev_status, void *stream);

/*
 * kvf32_decode_attn -- decode attention of the fp32 query over the fp32 cache:
 * s_t = sm_scale * q . k_t, softmax with a running maximum, fp32 accumulation
 * of v_t, split over the context and merged as in kvq8_decode_attn (one divide
 * by the summed weights at the end).  Workspace: kvq8_decode_workspace_bytes
 * (...) for the same sizes.  Other arguments as kvq8_decode_attn.
 */
kvq8_status kvf32_decode_attn(const float *q, int batch, int nqh, int nkv, int hd,
                              const float *k_cache, const float *v_cache,
                              int num_blocks, const int32_t *block_table,
                              int max_blocks, int block_size,
                              const int32_t *ctx_lens, float sm_scale,
                              float *out, void *workspace, size_t workspace_bytes,
                              uint32_t *dev_status, void *stream);

/* ------------------------------------------- decode without allocation --- */

/* Size of the static device scratch kvq8_decode_attn_noalloc uses (16 MiB). */
#define KVQ8_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * kvq8_decode_attn_noalloc -- kvq8_decode_attn for callers that cannot
 * allocate device memory.  The pages have no counterpart: this entry point
 * exists for library users who are given only their inputs, outputs and a
 * stream (plugin hosts that own the allocator, paths where cudaMalloc would
 * synchronise the device or is forbidden), and so cannot pass a workspace.
 *
 * Same arguments and results as kvq8_decode_attn, without the workspace: the
 * split partial results go to a static device array of
 * KVQ8_NOALLOC_SCRATCH_BYTES that every GPU which loads the library holds
 * until the process exits.  The call allocates nothing.
 *   - Arguments are checked exactly as kvq8_decode_attn checks them, in the
 *     same order; then sizes whose kvq8_decode_workspace_bytes(...) exceeds
 *     KVQ8_NOALLOC_SCRATCH_BYTES are rejected with KVQ8_ERR_WORKSPACE.  Every
 *     error returns before anything is enqueued.
 *   - The first call on a device that passes these checks looks up the
 *     array's device address (cudaGetSymbolAddress, with that device
 *     current) and remembers it for that device; make that first call before
 *     any stream capture on the device.  The address belongs to the device's
 *     context of that moment: after a cudaDeviceReset of the device, do not
 *     call this entry point again in the same process.
 *   - All calls share the one array and leave their partial results in it; no
 *     part of it needs to start at zero, since a call writes every record it
 *     reads, so the results equal kvq8_decode_attn's bit for bit.  Calls that
 *     overlap on the GPU (other streams, other threads) race on it: serialise
 *     them.
 */
kvq8_status kvq8_decode_attn_noalloc(const float *q, int batch, int nqh, int nkv, int hd,
                                     const int8_t *k_pool, const int8_t *v_pool,
                                     const float *k_scale, const float *v_scale,
                                     int num_blocks, const int32_t *block_table,
                                     int max_blocks, int block_size,
                                     const int32_t *ctx_lens, float sm_scale,
                                     float *out, uint32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ8_H */
