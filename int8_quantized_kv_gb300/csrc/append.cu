// append.cu -- quantise-append of new K/V rows into the paged INT8 cache, and
// the stand-alone 32-block query quantiser.
//
// Quantisation rule: [Day 9-3] §2 and [Day 9-1] §2 (kv_quantize_per_head):
// one fp32 scale = max|v|/127 per (token, kv head) row of 128 values, codes
// round_half_even(v/scale) in [-127, 127]; a row holding a NaN or an infinity
// (outside the rule) is stored as a row of zeros and flagged.
//
// Bulk append: one warp per run of 16 consecutive new tokens of one (sequence,
// kv head), with no shared memory and no block barrier, so that warps stream
// independently.  A row is one coalesced 512-byte read, a float4 per lane
// (lane l holds dims 4l..4l+3); the warp keeps the copies of its next five
// rows in flight to a shared-memory ring while it quantises.  K codes go straight to the token-major K tile
// (one 128-byte row, its 16-byte chunks permuted by slot).  For V each lane
// gathers the codes of its 4 dims over the 16 tokens in registers and writes
// them as one 16-byte piece of each dim-major row of the quarter.  A decode
// step's single token per sequence takes a warp per (sequence, kv head).
#include <limits.h>

#include "kvq8_device.cuh"
#include "kvq8_internal.cuh"
#include "kvq8_ptx.cuh"

namespace kvq8 {
namespace {

constexpr int kAppendWarps = 8;                  // one-token kernel: warps per CTA
// Bulk kernel: one warp per CTA.  A CTA decodes about 4 us of work, so the
// grid's tail (the last CTAs, each unable to draw an SM's share of the
// bandwidth alone) is short: 57.6 -> 55.7 us at 8 x 4096 tokens against CTAs
// of four warps (one quarter), whose tail was four times longer.
constexpr int kBulkWarps = 1;
constexpr int kQTok = kStageTok;                 // the V layout's 64-token quarter
constexpr int kRunTok = 16;                      // tokens per bulk warp
constexpr int kRunsPerQuarter = kQTok / kRunTok;
constexpr int kRing = 6;                         // rows per bulk warp staged in shared memory

// Position of the first new token of sequence b.
__device__ __forceinline__ int start_position(const AppendParams &p, int b) { return p.start_pos[b]; }

// Rows [vlo, vhi) of quarter x (counted from the quarter of start) of
// sequence b that the append writes, with qpos the quarter's first position;
// false when there are none.  Positions outside the table are left out, and
// flagged by the threads that pass `flag`.
__device__ __forceinline__ bool quarter_rows(const AppendParams &p, int b, long long x, int cap,
                                             bool flag, long long &start, long long &qpos,
                                             long long &vlo, long long &vhi) {
    const int s0 = start_position(p, b);
    start = s0;
    const long long q0 = start >= 0 ? start / kQTok : -((-start + kQTok - 1) / kQTok);
    qpos = (q0 + x) * kQTok;
    const long long lo = max(start, qpos);
    const long long hi = min(start + p.n_new, qpos + kQTok);
    if (lo >= hi) return false;
    if (lo < 0 || hi > cap) {
        if (flag) flag_status(p.dev_status, KVQ8_DEV_BAD_POSITION);
        if (hi <= 0 || lo >= cap) return false;
    }
    vlo = max(lo, 0LL);
    vhi = min(hi, (long long)cap);
    return true;
}

// Source offset (in floats) of the new row at position pos of (b, h).
__device__ __forceinline__ size_t new_row_offset(const AppendParams &p, int b, int h,
                                                 long long pos, long long start) {
    return (((size_t)b * p.n_new + (size_t)(pos - start)) * p.nkv + h) * kHD;
}

// Bulk append, one warp per task w = ((b * quarters + x) * nkv + h) * 4 + j:
// tokens 16j..16j+15 of quarter x (counted from the quarter of the first new
// token) of sequence b, kv head h.  The four runs of a quarter are consecutive
// CTAs, dispatched together, so that the 16-byte pieces of each V row are all
// written at about the same time.
__global__ void __launch_bounds__(kBulkWarps * 32, 32 / kBulkWarps)
quantize_append_kernel(AppendParams p, int quarters, long long tasks) {
    __shared__ __align__(16) float4 ring[kBulkWarps][kRing][2][32];   // [warp][slot][K, V][lane]

    // a programmatic dependent of the kernel before it, whose outputs it may
    // read: it waits for it first; the next kernel of the stream may be
    // scheduled now (it waits for this grid before it reads what it writes)
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long task = (long long)blockIdx.x * kBulkWarps + (threadIdx.x >> 5);
    if (task >= tasks) return;
    const int j = (int)(task % kRunsPerQuarter);
    long long t = task / kRunsPerQuarter;
    const int h = (int)(t % p.nkv);
    t /= p.nkv;
    const long long x = t % quarters;
    const int b = (int)(t / quarters);
    const int cap = p.max_blocks * kBS;
    long long start, qpos, vlo, vhi;
    if (!quarter_rows(p, b, x, cap, lane == 0 && j == 0, start, qpos, vlo, vhi)) return;
    const long long r0 = qpos + kRunTok * j;                    // first position of the run
    const long long lo = max(vlo, r0), hi = min(vhi, r0 + kRunTok);
    if (lo >= hi) return;                                        // warp-uniform
    const int phys = p.block_table[(size_t)b * p.max_blocks + (int)(qpos / kBS)];
    if (phys < 0 || phys >= p.num_blocks) {
        if (lane == 0) flag_status(p.dev_status, KVQ8_DEV_BAD_BLOCK_ID);
        return;
    }
    const size_t tile = (size_t)phys * p.nkv + h;
    const int slot0 = (int)(qpos % kBS) + kRunTok * j;          // a multiple of 16
    // K row of slot slot0 + r: its 16-byte chunk c sits at chunk position c ^ (r & 7)
    unsigned char *krow = reinterpret_cast<unsigned char *>(p.k_pool) + (tile * kBS + slot0) * kHD;
    // V: dim d of the run at vrun[d * 64 + r]
    int8_t *vrun = p.v_pool + tile * kHD * kBS + (size_t)(slot0 / kQTok) * kTileVQuarter + slot0 % kQTok;
    const int kchunk = lane >> 2, kword = lane & 3;

    if (lo == r0 && hi == r0 + kRunTok) {
        // the whole run: rows r0 .. r0 + 15 through a ring of kRing row slots in
        // shared memory, kRing - 1 rows in flight; each lane copies and later
        // reads back only its own 16 bytes of a row, so its own copy groups
        // order everything and the warp needs no barrier
        const size_t src = new_row_offset(p, b, h, r0, start);
        const float4 *kp = reinterpret_cast<const float4 *>(p.k_new + src) + lane;  // next row to copy
        const float4 *vp = reinterpret_cast<const float4 *>(p.v_new + src) + lane;
        const size_t step = (size_t)p.nkv * (kHD / 4);           // one row, in float4
        float4 (*slots)[2][32] = ring[threadIdx.x >> 5];
#pragma unroll
        for (int r = 0; r < kRing - 1; ++r) {
            cp_async16_cg(&slots[r][0][lane], kp);
            cp_async16_cg(&slots[r][1][lane], vp);
            cp_async_commit();
            kp += step;
            vp += step;
        }
        int rd = 0, wr = kRing - 1;    // slots of the row read next and the row copied next
        // groups of 4 rows; after group g, vw[i][3] holds its tokens of dim
        // 4 * lane + i and vw[i][0..2] the three groups before
        uint32_t vw[4][kRunTok / 4];
        float sc_keep = 0.0f;          // lane r < 16: K scale of row r; lane 16 + r: V scale
#pragma unroll 1
        for (int g = 0; g < kRunTok / 4; ++g) {
            uint32_t wg[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = 4 * g + u;
                cp_async_wait<kRing - 2>();   // row r has landed (rows r + 1 .. r + kRing - 2 may not)
                const float4 xks = slots[rd][0][lane], xvs = slots[rd][1][lane];
                rd = rd + 1 == kRing ? 0 : rd + 1;
                if (r + kRing - 1 < kRunTok) {   // into the slot of row r - 1, read before
                    cp_async16_cg(&slots[wr][0][lane], kp);
                    cp_async16_cg(&slots[wr][1][lane], vp);
                    kp += step;
                    vp += step;
                    wr = wr + 1 == kRing ? 0 : wr + 1;
                }
                cp_async_commit();               // possibly empty: one group per row
                float4 xk = xks, xv = xvs;
                const float sk = kv_row_scale_checked(xk, p.dev_status);
                const float sv = kv_row_scale_checked(xv, p.dev_status);
                const uint32_t wk = low_bytes4(kv_code_bytes4(xk, sk));
                const uint4 cv = kv_code_bytes4(xv, sv);
                reinterpret_cast<uint32_t *>(krow + r * kHD + ((kchunk ^ (r & 7)) << 4))[kword] = wk;
                if (lane == r) sc_keep = sk;
                if (lane == 16 + r) sc_keep = sv;
                // byte u of the group's word of each of the lane's dims
                constexpr uint32_t kIns[4] = {0x3210, 0x3240, 0x3410, 0x4210};
                if (u == 0) {
                    wg[0] = cv.x; wg[1] = cv.y; wg[2] = cv.z; wg[3] = cv.w;
                } else {
                    wg[0] = __byte_perm(wg[0], cv.x, kIns[u]);
                    wg[1] = __byte_perm(wg[1], cv.y, kIns[u]);
                    wg[2] = __byte_perm(wg[2], cv.z, kIns[u]);
                    wg[3] = __byte_perm(wg[3], cv.w, kIns[u]);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                vw[i][0] = vw[i][1];
                vw[i][1] = vw[i][2];
                vw[i][2] = vw[i][3];
                vw[i][3] = wg[i];
            }
        }
        (lane < 16 ? p.k_scale : p.v_scale)[tile * kBS + slot0 + (lane & 15)] = sc_keep;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4 *>(vrun + (size_t)(4 * lane + i) * kQTok) =
                make_uint4(vw[i][0], vw[i][1], vw[i][2], vw[i][3]);
    } else {
        // part of a run (the ends of the appended range): row by row
        for (int r = (int)(lo - r0); r < (int)(hi - r0); ++r) {
            const size_t src = new_row_offset(p, b, h, r0 + r, start);
            float4 xk = reinterpret_cast<const float4 *>(p.k_new + src)[lane];
            float4 xv = reinterpret_cast<const float4 *>(p.v_new + src)[lane];
            const float sk = kv_row_scale_checked(xk, p.dev_status);
            const float sv = kv_row_scale_checked(xv, p.dev_status);
            reinterpret_cast<uint32_t *>(krow + r * kHD + ((kchunk ^ (r & 7)) << 4))[kword] =
                low_bytes4(kv_code_bytes4(xk, sk));
            const uint4 cv = kv_code_bytes4(xv, sv);
            vrun[(size_t)(4 * lane + 0) * kQTok + r] = (int8_t)cv.x;
            vrun[(size_t)(4 * lane + 1) * kQTok + r] = (int8_t)cv.y;
            vrun[(size_t)(4 * lane + 2) * kQTok + r] = (int8_t)cv.z;
            vrun[(size_t)(4 * lane + 3) * kQTok + r] = (int8_t)cv.w;
            if (lane == 0) {
                p.k_scale[tile * kBS + slot0 + r] = sk;
                p.v_scale[tile * kBS + slot0 + r] = sv;
            }
        }
    }
}

// One new token per sequence (n_new == 1): a warp per (sequence, kv head), K
// row and V row quantised from one float4 per lane; no staging needed.  (A
// decode step appends inside its split kernel instead.)
__global__ void __launch_bounds__(kAppendWarps * 32)
quantize_append_token_kernel(AppendParams p) {
    // Launched as a programmatic dependent: wait for the previous kernel in the
    // stream (which may have produced the new token's K and V), then let the
    // next kernel of the step be scheduled.
    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wid = blockIdx.x * kAppendWarps + warp;
    if (wid >= p.batch * p.nkv) return;
    const int b = wid / p.nkv, h = wid % p.nkv;
    const int cap = p.max_blocks * kBS;
    const int pos = start_position(p, b);
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
    float4 xk = reinterpret_cast<const float4 *>(p.k_new + src)[lane];
    float4 xv = reinterpret_cast<const float4 *>(p.v_new + src)[lane];
    {
        const float s = kv_row_scale_checked(xk, p.dev_status);
        unsigned char *row = reinterpret_cast<unsigned char *>(p.k_pool) + (tile * kBS + slot) * kHD;
        reinterpret_cast<uint32_t *>(row + (((lane >> 2) ^ (slot & 7)) << 4))[lane & 3] =
            low_bytes4(kv_code_bytes4(xk, s));
        if (lane == 0) p.k_scale[tile * kBS + slot] = s;
    }
    {
        const float s = kv_row_scale_checked(xv, p.dev_status);
        int8_t *vg = p.v_pool + tile * kHD * kBS + (size_t)(slot / kStageTok) * kTileVQuarter + slot % kStageTok;
        const uint4 c = kv_code_bytes4(xv, s);
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
    // (kvq8_quantize_q has no status word: a non-finite block is zeroed unflagged)
    quantize_q_row_warp(q + row * kHD, threadIdx.x & 31, codes + row * kHD, scales + row * kNQB, nullptr);
}

}  // namespace

cudaError_t launch_quantize_append(const AppendParams &p, cudaStream_t s) {
    if (p.n_new == 1) {
        const int64_t warps = (int64_t)p.batch * p.nkv;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)((warps + kAppendWarps - 1) / kAppendWarps));
        cfg.blockDim = dim3(kAppendWarps * 32);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, quantize_append_token_kernel, p);
    } else {
        // quarters touched by n_new consecutive positions: at most n_new/64 + 1
        const int quarters = p.n_new / kQTok + (p.n_new % kQTok ? 2 : 1);
        const long long tasks = (long long)kRunsPerQuarter * quarters * p.nkv * p.batch;
        const long long blocks = (tasks + kBulkWarps - 1) / kBulkWarps;
        if (blocks > INT_MAX) return cudaErrorInvalidConfiguration;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(kBulkWarps * 32);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, quantize_append_kernel, p, quarters, tasks);
    }
}

cudaError_t launch_quantize_q(const float *q, int64_t n_rows, int8_t *codes, float *scales,
                              cudaStream_t s) {
    const int64_t blocks = (n_rows + 3) / 4;
    quantize_q_kernel<<<(unsigned)blocks, 128, 0, s>>>(q, n_rows, codes, scales);
    return cudaGetLastError();
}

}  // namespace kvq8
