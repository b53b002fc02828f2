// decode.cu -- single-query decode attention over the paged INT8 cache:
// a persistent split-KV kernel and the merge of its partial results.
//
// Method: [Day 9-2] "flash_attn_single_q_q8_neon" §1-§3.  The query heads that
// share a kv head are quantised once in 32-blocks (segment 1); every cached
// token's score is rebuilt from exact int32 block dots times the query block
// scales, times the token's K scale and the softmax scale (segment 2, "three
// key points"); the softmax runs online with a running maximum, rescaling the
// running sum and the V accumulator when the maximum grows; V enters as
// int8 code * (weight * V scale) with fp32 accumulation; one division by the
// sum at the end (segment 3).  The softmax runs in base 2 (scores are
// pre-multiplied by log2(e)), which leaves the normalised weights unchanged.
//
// GB300 structure of the split kernel (one CTA per SM, 8 warps; for G = 2 and
// a call of at least 16 units two CTAs per SM, each with half the ring and at
// most 128 registers a thread, see kSmemLimit2):
//  * Work: the cache is a sequence of 64-token stages, unit by unit (unit =
//    (sequence, kv head)); CTA c takes stages [c*T/C, (c+1)*T/C), i.e. an
//    equal share regardless of how ragged the contexts are.  Where a unit
//    starts or ends inside the range, the CTA emits one partial record for
//    that (CTA, unit) segment.
//  * Warp 7 is the producer: for every stage it issues four 1-D bulk copies
//    (K 8 KiB, V 8 KiB, two 256 B scale runs) into a ring of shared-memory
//    slots, tracked by full/empty mbarriers.  The KV stream uses an L2
//    evict-first policy: it is read exactly once.
//  * Warps 0..6 take the stages of a segment round-robin (a fixed assignment,
//    so results are reproducible bit for bit), each with its own
//    online-softmax state (two warps per SM sub-partition leave room for 255
//    registers a thread).  Q.K: lane = token (two tokens per lane), dp4a on
//    int8 codes, exact int32 per 32-block.  P.V: tensor-core MMA m16n8k16 with
//    A = V (int8 codes + 128 as exact fp16 subnormals, the offset removed
//    once per stage by a correction tile) and B = P, the weights times the V
//    scale, split into fp16 high + low parts and scaled per stage by a power
//    of two so that fp16 range and precision lose nothing that fp32
//    accumulation keeps; D accumulates in fp32.
//  * At the end of a segment the 7 warp states are merged in shared memory
//    and written as one record per query head.
// All waits are bounded: a wait that times out sets KVQ8_DEV_TIMEOUT and the
// CTA unwinds without leaving copies in flight.  The kernel is launched as a
// programmatic dependent of the previous kernel in its stream, so that its
// launch overlaps that kernel; every thread waits for that kernel's results
// first.  The combine releases the next kernel of the stream as soon as the
// split's records are visible to it.  In a decode step the split kernel also
// appends the step's new token: the consumer that decodes the stage holding
// position ctx_lens[b] - 1 quantises the token into that staged stage and
// into the pools (no separate append launch).
#include <cuda_fp16.h>
#include <math.h>

#include "kvq8_device.cuh"
#include "kvq8_internal.cuh"
#include "kvq8_ptx.cuh"

namespace kvq8 {
namespace {

constexpr int kConsumerWarps = 7;
constexpr int kSplitThreads = (kConsumerWarps + 1) * 32;
constexpr int kSmemLimit = 232448;          // 227 KiB opt-in per CTA on sm_103a
// In a mixed-precision decode the int8 split runs after the 4-bit split of the
// same call and takes each SM as that grid leaves it.  With a ring this small
// (and its registers) it fits beside one CTA of the 4-bit split (about 48 KiB
// of an SM's 228 KiB), so it starts on an SM as soon as two of its three
// 4-bit CTAs are done, instead of waiting for the last, which would run
// alone with a third of the SM's warps.
constexpr int kSmemLimitMixed = 184320;
// Two CTAs per SM (G = 2, calls of at least 16 units, and the int8 part of a
// G = 2 mixed-precision decode): each gets half of the SM's 228 KiB less the
// per-CTA reserve (a 6-stage ring) and at most 128 registers a thread (the
// G = 2 consumer fits with 4 bytes spilled).  The 14 consumer warps of an SM
// then hide more of each stage's latency: the 28-layer 8K step streams at 96 %
// of the copy peak instead of 95 %.  Such a CTA also fits beside one CTA of
// the 4-bit split.  A call of fewer units keeps one CTA per SM: with twice the
// CTAs a unit's record count would pass what the merge reads in one round, and
// a few-unit call is latency-bound.
constexpr int kSmemLimit2 = 115712;
constexpr int kTwoPerSmMinUnits = 16;
constexpr int kTwoPerSmMinStages = 16;   // per CTA, counted on the table's width
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;
constexpr int kPRowHalves = 72;             // P row: 64 tokens + 8 halves of padding
constexpr float kLazyLog2 = 8.0f;           // running-max slack (log2 units), see segment 2b

template <int G, int kLimit = kSmemLimit>
struct SplitLayout {
    // per consumer warp: P (hi, lo) [G][72] halves during a stage, or the
    // warp's final state (acc [G][128], M [G], S [G]) when a segment ends
    static constexpr int kScratch = ((G * 520) + 15) / 16 * 16;
    static constexpr int kQCodes = G * kHD;
    static constexpr int kQScale = G * kNQB * 4;
    static constexpr int kMisc = 128;
    static constexpr int kFixed = kConsumerWarps * kScratch + kQCodes + kQScale + kMisc;
    static constexpr int kStages = (kLimit - kFixed - 512) / (kStageBytes + 16 + 16 + 4);
    static constexpr int oRing = 0;
    static constexpr int oScratch = kStages * kStageBytes;
    static constexpr int oQCodes = oScratch + kConsumerWarps * kScratch;
    static constexpr int oQScale = oQCodes + kQCodes;
    static constexpr int oMisc = oQScale + kQScale;
    static constexpr int oFull = oMisc + kMisc;
    static constexpr int oEmpty = oFull + kStages * 8;
    static constexpr int oSkip = oEmpty + kStages * 8;
    static constexpr int oDone = oSkip + kStages * 4;
    static constexpr int kBytes = oDone + kStages * 4;
    static_assert(oMisc % 16 == 0 && oFull % 16 == 0 && oScratch % 16 == 0, "alignment");
    static_assert(kBytes <= kLimit, "shared memory budget");
    static_assert(kStages >= 6, "ring too shallow");
    static_assert(G * 2 * kPRowHalves * 2 <= kScratch, "P fits the warp scratch");
};

struct Misc {
    long long warp_tot[kSplitThreads / 32];
    long long base;   // stage prefix at the first unit of sequence b0
    int b0;
};

__device__ __forceinline__ int clamp_len(int L, int cap) { return max(0, min(L, cap)); }

// The tokens [x, y) of sequence b that this launch decodes: [0, L) normally;
// [256 * first_q8_block[b], L) when the older blocks of the sequence are held
// in the 4-bit cache (mixed precision by token age; kMixed).
template <bool kMixed = true>
__device__ __forceinline__ int2 seq_span(const DecodeParams &p, int b, int cap) {
    const int L = clamp_len(p.ctx_lens[b], cap);
    const int s = (kMixed && p.first_q8_block) ? min(L, max(0, min(p.first_q8_block[b], cap / kBS)) * kBS) : 0;
    return make_int2(s, L);
}
__device__ __forceinline__ int span_stages(int2 sp) { return (sp.y - sp.x + kStageTok - 1) / kStageTok; }

// int8 codes v of 4 consecutive tokens -> two fp16 pairs (tokens 0,1 and 2,3)
// holding (v + 128) * 2^-24: the offset byte in the low bits of a half is the
// fp16 subnormal of that value (exact; the tensor cores take subnormals as
// they are).  The offset is removed by kNegOffset below.
__device__ __forceinline__ void codes_to_sub2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t x = w ^ 0x80808080u;
    lo = __byte_perm(x, 0u, 0x4140);
    hi = __byte_perm(x, 0u, 0x4342);
}
// fp16 pair (-2^-17, -2^-17) = -128 code steps of 2^-24: an A operand of these
// times P gives -128 * 2^-24 * sum_t P[t][col] in every row, the offset's
// share of the accumulator for that stage.
constexpr uint32_t kNegOffset = 0x80808080u;
constexpr float kCodeUnit = 16777216.0f;   // 2^24: one code step of codes_to_sub2

__device__ __forceinline__ int4 lds128(const void *p) { return *reinterpret_cast<const int4 *>(p); }

// Warp-wide maxima in one redux instruction.  Floats are mapped to integers
// whose signed order is the float order (negative values get their magnitude
// bits flipped), reduced, and mapped back.
__device__ __forceinline__ int redux_max_i32(int v) { return __reduce_max_sync(0xffffffffu, v); }

__device__ __forceinline__ float redux_max_f32(float x) {
    int k = __float_as_int(x);
    k ^= (k >> 31) & 0x7fffffff;
    k = __reduce_max_sync(0xffffffffu, k);
    k ^= (k >> 31) & 0x7fffffff;
    return __int_as_float(k);
}

// Waits until *done reaches `round` (the slot's earlier stages are consumed);
// false after timeout_ns.
__device__ __forceinline__ bool slot_turn_bounded(volatile int *done, int round, uint64_t timeout_ns) {
    if (*done >= round) return true;
    const uint64_t t0 = global_timer_ns();
    while (*done < round) {
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
    return true;
}

// A decode step's new token of unit (b, h), position pos = ctx_lens[b] - 1,
// which is row t of the stage staged at st (xk, xv: the token's K and V rows,
// lane l holding dims 4l..4l+3, and phys: the id of the cache block holding
// pos, all loaded by the caller ahead of time; phys = -1: loaded here):
// quantised by the warp ([Day 9-3] §2 rule, the same functions as the append
// kernels), written over the row the copy brought in (K row with its chunk
// order, V column of the dim-major quarter, both scales) and into the pools
// and scale arrays.  Only this CTA reads that position in this launch.  The
// block id is valid: the stage was copied.
__device__ __noinline__ void append_new_token(const DecodeParams &p, int b, int h, int pos, int t,
                                                 int lane, unsigned char *st, float4 xk, float4 xv, int phys) {
    if (phys < 0) phys = p.block_table[(size_t)b * p.max_blocks + pos / kBS];
    const float sk = kv_row_scale_checked(xk, p.dev_status), sv = kv_row_scale_checked(xv, p.dev_status);
    const uint32_t wk = low_bytes4(kv_code_bytes4(xk, sk));
    const uint4 cv = kv_code_bytes4(xv, sv);
    const int slot = pos % kBS;   // slot & 7 == t & 7: stages start at multiples of 64
    const int kpos = ((((lane >> 2) ^ (slot & 7)) << 4) + (lane & 3) * 4);
    // the staged stage
    *reinterpret_cast<uint32_t *>(st + t * kHD + kpos) = wk;
    unsigned char *vs = st + kStageKBytes + t;
    vs[(4 * lane + 0) * kStageTok] = (unsigned char)cv.x;
    vs[(4 * lane + 1) * kStageTok] = (unsigned char)cv.y;
    vs[(4 * lane + 2) * kStageTok] = (unsigned char)cv.z;
    vs[(4 * lane + 3) * kStageTok] = (unsigned char)cv.w;
    float *scl = reinterpret_cast<float *>(st + kStageKBytes + kStageVBytes);
    // the cache (the pools of a decode step are the caller's writable buffers)
    const size_t tile = (size_t)phys * p.nkv + h;
    int8_t *kp = const_cast<int8_t *>(p.k_pool), *vp = const_cast<int8_t *>(p.v_pool);
    *reinterpret_cast<uint32_t *>(kp + (tile * kBS + slot) * kHD + kpos) = wk;
    int8_t *vg = vp + tile * kHD * kBS + (size_t)(slot / kStageTok) * kTileVQuarter + slot % kStageTok;
    vg[(size_t)(4 * lane + 0) * kStageTok] = (int8_t)cv.x;
    vg[(size_t)(4 * lane + 1) * kStageTok] = (int8_t)cv.y;
    vg[(size_t)(4 * lane + 2) * kStageTok] = (int8_t)cv.z;
    vg[(size_t)(4 * lane + 3) * kStageTok] = (int8_t)cv.w;
    if (lane == 0) {
        scl[t] = sk;
        scl[kStageTok + t] = sv;
        const_cast<float *>(p.k_scale)[tile * kBS + slot] = sk;
        const_cast<float *>(p.v_scale)[tile * kBS + slot] = sv;
    }
    __syncwarp();   // the patched rows are read by every lane below
}

// The ring and register budget of a split-kernel instantiation: a two-per-SM
// grid, a mixed decode's int8 split, or the default.
template <int G, bool kMixed, int kCtas>
using SplitLay = SplitLayout<G, kCtas == 2 ? kSmemLimit2 : (kMixed ? kSmemLimitMixed : kSmemLimit)>;

template <int G, bool kMixed, int kCtas>
__global__ void __launch_bounds__(kSplitThreads, kCtas)
decode_split_kernel(DecodeParams p) {
    using Lay = SplitLay<G, kMixed, kCtas>;
    extern __shared__ __align__(1024) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int cap = p.max_blocks * kBS;
    // Launched as a programmatic dependent of the previous kernel in the stream
    // (its launch overlaps that kernel's end), whose outputs may be this
    // kernel's inputs: every thread waits for it here first -- unless the
    // caller vouches that the cache, the block table and the context lengths
    // were final before that kernel began (cache_ready): then the prologue and
    // the producer's copies go ahead, and only the consumers wait (they read
    // the query and the new token and write the workspace).
    // In a mixed-precision decode (kMixed) the kernel before is the 4-bit split
    // of the same call, which writes nothing this kernel reads (it released
    // this one right after its own wait): no wait here; this kernel waits for
    // it at its end instead, before completing.
    if (!kMixed && !p.cache_ready) pdl_wait();
    Misc *misc = reinterpret_cast<Misc *>(smem + Lay::oMisc);
    int8_t *q_codes = reinterpret_cast<int8_t *>(smem + Lay::oQCodes);
    float *q_scale = reinterpret_cast<float *>(smem + Lay::oQScale);
    volatile int *skip = reinterpret_cast<volatile int *>(smem + Lay::oSkip);
    // done[s] = how many stages of slot s have been consumed.  A consumer waits
    // on a slot's full barrier only once the slot's previous stage is consumed,
    // so every wait targets the barrier's current phase (a parity wait cannot
    // tell a phase two rounds ahead from the previous one).
    volatile int *done = reinterpret_cast<volatile int *>(smem + Lay::oDone);
    const uint32_t full0 = smem_addr(smem + Lay::oFull), empty0 = smem_addr(smem + Lay::oEmpty);

    // ---- prologue: total stage count T and where this CTA's range starts ----
    const int per = (p.batch + kSplitThreads - 1) / kSplitThreads;
    const int b_lo = min(p.batch, tid * per), b_hi = min(p.batch, b_lo + per);
    // the first context length is loaded before the barriers are initialised,
    // so that its latency covers them
    const int L_first = b_lo < b_hi ? p.ctx_lens[b_lo] : 0;
    if (tid < Lay::kStages) {
        mbar_init(full0 + 8 * tid, 1);
        mbar_init(empty0 + 8 * tid, 1);
        done[tid] = 0;
        fence_mbar_init();
    }
    long long mine = 0;
    for (int b = b_lo; b < b_hi; ++b) {
        const int L = b == b_lo ? L_first : p.ctx_lens[b];
        if (c == 0 && (L < 0 || L > cap)) flag_status(p.dev_status, KVQ8_DEV_BAD_CTX_LEN);
        mine += (long long)p.nkv * span_stages(seq_span<kMixed>(p, b, cap));
    }
    long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) misc->warp_tot[warp] = incl;
    __syncthreads();
    if (tid == 0) {
        long long run = 0;
        for (int w = 0; w < kSplitThreads / 32; ++w) {
            const long long t = misc->warp_tot[w];
            misc->warp_tot[w] = run;
            run += t;
        }
        misc->base = run;  // temporarily: T
    }
    __syncthreads();
    const long long T = misc->base;
    const long long excl = misc->warp_tot[warp] + incl - mine;
    // the stages are shared by min(gridDim.x, T) CTAs so that every active CTA
    // owns at least one stage and the CTAs covering a unit are consecutive
    const int C = (int)min((long long)gridDim.x, T);
    // lo = c*T/C and hi = (c+1)*T/C from one 64-bit division: with T = Tq*C + Tr,
    // k*T/C = k*Tq + (k*Tr)/C exactly, and k*Tr < C*C fits 32 bits
    long long lo = 0, hi = 0;
    if (c < C) {
        const long long Tq = T / C;
        const int Tr = (int)(T - Tq * C);
        lo = (long long)c * Tq + (c * Tr) / C;
        hi = (long long)(c + 1) * Tq + ((c + 1) * Tr) / C;
    }
    __syncthreads();
    if (mine > 0 && excl <= lo && lo < excl + mine) {
        long long acc = excl;
        for (int b = b_lo; b < b_hi; ++b) {
            const long long n = (long long)p.nkv * span_stages(seq_span<kMixed>(p, b, cap));
            if (lo < acc + n) {
                misc->b0 = b;
                misc->base = acc;
                break;
            }
            acc += n;
        }
    }
    __syncthreads();

    int b = 0, h = 0, off = 0;
    if (hi > lo) {
        b = misc->b0;
        const int nb = span_stages(seq_span<kMixed>(p, b, cap));
        const long long rel = lo - misc->base;   // < nkv * nb
        if (rel <= 0x7fffffffLL) {
            h = (int)rel / nb;
            off = (int)rel - h * nb;
        } else {
            h = (int)(rel / nb);
            off = (int)(rel % nb);
        }
    }

    if (warp == kConsumerWarps) {
        // =========================== producer warp ===========================
        const uint64_t pol = l2_evict_first_policy();
        bool aborted = false;
        long long remaining = hi - lo;
        int kbase = 0;
        while (remaining > 0 && b < p.batch) {
            const int2 sp = seq_span<kMixed>(p, b, cap);
            const int nb = span_stages(sp);
            if (nb == 0) { ++b; h = 0; off = 0; continue; }
            const int seg_n = (int)min((long long)(nb - off), remaining);
            const int32_t *row = p.block_table + (size_t)b * p.max_blocks;
            int tbl_base = -1, tbl_reg = -1;
            for (int j = 0; j < seg_n; ++j) {
                const int k = kbase + j, slot = k % Lay::kStages;
                const uint32_t par = ((k / Lay::kStages) & 1) ^ 1;
                const int t0 = sp.x + (off + j) * kStageTok;
                const int lb = t0 / kBS, quarter = (t0 / kStageTok) & 3;
                if (tbl_base < 0 || lb >= tbl_base + 32) {
                    tbl_base = lb;
                    tbl_reg = (lb + lane < p.max_blocks) ? row[lb + lane] : -1;
                }
                const int phys = __shfl_sync(0xffffffffu, tbl_reg, lb - tbl_base);
                if (lane == 0) {
                    const uint32_t fb = full0 + 8 * slot;
                    if (!aborted && !mbar_wait_bounded(empty0 + 8 * slot, par, kWaitTimeoutNs)) {
                        aborted = true;
                        flag_status(p.dev_status, KVQ8_DEV_TIMEOUT);
                    }
                    if (aborted) {
                        // leave the slot unfilled; its consumer times out and unwinds
                    } else if (phys >= 0 && phys < p.num_blocks) {
                        skip[slot] = 0;
                        const size_t tile = (size_t)phys * p.nkv + h;
                        unsigned char *st = smem + Lay::oRing + (size_t)slot * kStageBytes;
                        mbar_arrive_expect_tx(fb, kStageBytes);
                        bulk_copy_g2s(smem_addr(st), p.k_pool + (tile * kBS + quarter * kStageTok) * kHD,
                                      kStageKBytes, fb, pol);
                        bulk_copy_g2s(smem_addr(st + kStageKBytes),
                                      p.v_pool + tile * kHD * kBS + quarter * kTileVQuarter,
                                      kStageVBytes, fb, pol);
                        bulk_copy_g2s(smem_addr(st + kStageKBytes + kStageVBytes),
                                      p.k_scale + tile * kBS + quarter * kStageTok, kStageSBytes, fb, pol);
                        bulk_copy_g2s(smem_addr(st + kStageKBytes + kStageVBytes + kStageSBytes),
                                      p.v_scale + tile * kBS + quarter * kStageTok, kStageSBytes, fb, pol);
                    } else {
                        skip[slot] = 1;
                        flag_status(p.dev_status, KVQ8_DEV_BAD_BLOCK_ID);
                        mbar_arrive(fb);
                    }
                }
                __syncwarp();
            }
            remaining -= seg_n;
            kbase += seg_n;
            off = 0;
            if (++h == p.nkv) { h = 0; ++b; }
        }
        // no copy may still be in flight when the CTA exits
        if (lane == 0) {
            for (int k = max(0, kbase - Lay::kStages); k < kbase; ++k)
                mbar_wait_bounded(full0 + 8 * (k % Lay::kStages), (k / Lay::kStages) & 1, kWaitTimeoutNs);
        }
    } else {
        // =========================== consumer warps ==========================
        if (!kMixed && p.cache_ready) pdl_wait();
        unsigned char *scratch = smem + Lay::oScratch + warp * Lay::kScratch;
        __half *p_hi = reinterpret_cast<__half *>(scratch);
        __half *p_lo = p_hi + G * kPRowHalves;
        float *red_acc = reinterpret_cast<float *>(scratch);
        float *red_m = red_acc + G * kHD;
        float *red_s = red_m + G;
        const int n = lane >> 2, t4 = lane & 3;  // MMA fragment coordinates
        // P.V for G <= 4 packs P's high fp16 parts into columns 0..G-1 and its
        // low parts into G..2G-1 of one MMA (half the MMAs); the columns' sums
        // are added at the segment's end.  Accumulator columns 2*t4, 2*t4 + 1
        // then belong to heads col_head0, col_head1 (for their rescaling).
        constexpr bool kPackPV = G <= 4;
        const int col_head0 = kPackPV ? (2 * t4) % G : 2 * t4;
        const int col_head1 = kPackPV ? (2 * t4 + 1) % G : 2 * t4 + 1;
        bool aborted = false;
        long long remaining = hi - lo;
        int kbase = 0;
        // This warp's query rows (heads g = warp, warp + 7 of the unit) of the
        // unit (qb, qh), loaded one segment ahead so that the quantisation at
        // a segment's start waits for no global load.
        constexpr int kQRows = (G + kConsumerWarps - 1) / kConsumerWarps;
        float qx[kQRows][4];
        int qb = -1, qh = -1;
        auto load_q_rows = [&](int bb, int hh) {
#pragma unroll
            for (int i = 0; i < kQRows; ++i) {
                const int g = warp + i * kConsumerWarps;
                if (g < G) {
                    const float *r = p.q + ((size_t)bb * p.nqh + (size_t)hh * G + g) * kHD;
#pragma unroll
                    for (int k = 0; k < 4; ++k) qx[i][k] = r[32 * k + lane];
                }
            }
            qb = bb;
            qh = hh;
        };
        while (remaining > 0 && b < p.batch) {
            const int2 sp = seq_span<kMixed>(p, b, cap);
            const int L = sp.y;
            const int nb = span_stages(sp);
            if (nb == 0) { ++b; h = 0; off = 0; continue; }
            const int seg_n = (int)min((long long)(nb - off), remaining);
            const int u = b * p.nkv + h;
            // a decode step appends its new token at position ctx_lens[b] - 1
            // (none for an empty context or one beyond the table)
            int app_pos = -1;
            if (!kMixed && p.k_new) {   // (a mixed-precision decode appends nothing)
                const int Lraw = p.ctx_lens[b];
                if (Lraw >= 1 && Lraw <= cap) app_pos = Lraw - 1;
            }

            // the warp that decodes the stage holding the new token loads the
            // token's K and V rows and its block id now, beside the query rows,
            // so that their latencies overlap and none is left for the stage
            // (G = 8: at the stage, its registers are spent)
            constexpr bool kPreloadNew = G <= 4;
            float4 nxk = make_float4(0.f, 0.f, 0.f, 0.f), nxv = nxk;
            int nphys = -1;
            if (kPreloadNew && app_pos >= sp.x) {
                const int sj = (app_pos - sp.x) / kStageTok - off;
                if (sj >= 0 && sj < seg_n && sj % kConsumerWarps == warp) {
                    const size_t src = ((size_t)b * p.nkv + h) * kHD;
                    nxk = reinterpret_cast<const float4 *>(p.k_new + src)[lane];
                    nxv = reinterpret_cast<const float4 *>(p.v_new + src)[lane];
                    nphys = p.block_table[(size_t)b * p.max_blocks + app_pos / kBS];
                }
            }

            // segment 1: quantise this unit's G query heads once
            if (qb != b || qh != h) load_q_rows(b, h);   // not loaded ahead
            named_barrier_sync(1, kConsumerWarps * 32);
#pragma unroll
            for (int i = 0; i < kQRows; ++i) {
                const int g = warp + i * kConsumerWarps;
                if (g < G) quantize_q_vals_warp(qx[i], lane, q_codes + g * kHD, q_scale + g * kNQB, p.dev_status);
            }
            named_barrier_sync(1, kConsumerWarps * 32);
            if (remaining > seg_n) {   // the next segment's unit follows this one
                const int nh = h + 1 == p.nkv ? 0 : h + 1;
                const int nbq = h + 1 == p.nkv ? b + 1 : b;
                if (nbq < p.batch) load_q_rows(nbq, nh);
            }

            // this CTA holds the unit's first stage (off == 0): it publishes where
            // the unit's records are, CTAs c .. c_last (computed here, off the
            // path of the segment's end)
            int meta_n = 0;
            if (tid == 0 && off == 0) {
                const long long end_u = lo + kbase + nb;
                meta_n = (int)((end_u * C + T - 1) / T) - c;
            }
            float M[G], Sl[G], acc[8][4];
#pragma unroll
            for (int g = 0; g < G; ++g) { M[g] = -INFINITY; Sl[g] = 0.0f; }
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[mt][i] = 0.0f;
            int e_cur = 1000;  // acc holds values in units of 2^e_cur (first stage sets it)

            for (int j = warp; j < seg_n; j += kConsumerWarps) {
                const int k = kbase + j, slot = k % Lay::kStages, round = k / Lay::kStages;
                const uint32_t par = round & 1;
                if (!aborted && !slot_turn_bounded(done + slot, round, kWaitTimeoutNs)) aborted = true;
                if (!aborted && !mbar_wait_bounded(full0 + 8 * slot, par, kWaitTimeoutNs)) aborted = true;
                if (aborted && lane == 0) flag_status(p.dev_status, KVQ8_DEV_TIMEOUT);
                if (!aborted && !skip[slot]) {
                    const unsigned char *st = smem + Lay::oRing + (size_t)slot * kStageBytes;
                    const int8_t *kst = reinterpret_cast<const int8_t *>(st);
                    const int8_t *vst = kst + kStageKBytes;
                    const float *ks_st = reinterpret_cast<const float *>(st + kStageKBytes + kStageVBytes);
                    const float *vs_st = ks_st + kStageTok;
                    const int nvalid = min(kStageTok, L - (sp.x + (off + j) * kStageTok));
                    const int tnew = app_pos - (sp.x + (off + j) * kStageTok);
                    if (tnew >= 0 && tnew < kStageTok) {
                        if (!kPreloadNew) {
                            const size_t src = ((size_t)b * p.nkv + h) * kHD;
                            nxk = reinterpret_cast<const float4 *>(p.k_new + src)[lane];
                            nxv = reinterpret_cast<const float4 *>(p.v_new + src)[lane];
                        }
                        append_new_token(p, b, h, app_pos, tnew, lane, const_cast<unsigned char *>(st), nxk, nxv, nphys);
                    }
                    const int ta = lane, tb = lane + 32;
                    const bool va = ta < nvalid, vb = tb < nvalid;

                    // ---- segment 2a: int32 block dots, lane = token ----
                    int da[G][kNQB], db[G][kNQB];
#pragma unroll
                    for (int g = 0; g < G; ++g)
#pragma unroll
                        for (int q = 0; q < kNQB; ++q) { da[g][q] = 0; db[g][q] = 0; }
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const int4 ka = lds128(kst + ta * kHD + ((cc ^ (ta & 7)) << 4));
                        const int4 kb = lds128(kst + tb * kHD + ((cc ^ (tb & 7)) << 4));
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            const int4 qw = lds128(q_codes + g * kHD + cc * 16);
                            int x = da[g][cc >> 1], y = db[g][cc >> 1];
                            x = __dp4a(ka.x, qw.x, x); y = __dp4a(kb.x, qw.x, y);
                            x = __dp4a(ka.y, qw.y, x); y = __dp4a(kb.y, qw.y, y);
                            x = __dp4a(ka.z, qw.z, x); y = __dp4a(kb.z, qw.z, y);
                            x = __dp4a(ka.w, qw.w, x); y = __dp4a(kb.w, qw.w, y);
                            da[g][cc >> 1] = x;
                            db[g][cc >> 1] = y;
                        }
                    }
                    const float ksa = ks_st[ta], ksb = ks_st[tb];
                    const float vsa = va ? vs_st[ta] : 0.0f, vsb = vb ? vs_st[tb] : 0.0f;

                    // power-of-two unit of this stage's P: 2^e > max vs, so that
                    // p' = w * vs * 2^-e stays below 2^8 (w < 2^8, see below).  e only
                    // moves when it must grow or has become 2^12 too large.
                    const int e_need = redux_max_i32(
                        ((__float_as_int(fmaxf(vsa, vsb)) >> 23) & 0xff) - 126);  // 0 -> -126
                    int e = e_cur;
                    if (e_need > e_cur || e_need < e_cur - 12) e = max(-120, min(120, e_need));
                    const float inv = __int_as_float((127 - e) << 23);

                    // ---- segment 2b: scores, online softmax ----
                    float sa[G], sb[G];
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float4 qs = *reinterpret_cast<const float4 *>(q_scale + g * kNQB);
                        float a = (float)da[g][0] * qs.x;
                        a = fmaf((float)da[g][1], qs.y, a);
                        a = fmaf((float)da[g][2], qs.z, a);
                        a = fmaf((float)da[g][3], qs.w, a);
                        float bb = (float)db[g][0] * qs.x;
                        bb = fmaf((float)db[g][1], qs.y, bb);
                        bb = fmaf((float)db[g][2], qs.z, bb);
                        bb = fmaf((float)db[g][3], qs.w, bb);
                        sa[g] = va ? a * ksa * p.sm_scale_log2 : -INFINITY;
                        sb[g] = vb ? bb * ksb * p.sm_scale_log2 : -INFINITY;
                    }
                    // The running maximum M is raised only when a score exceeds it by
                    // more than 2^kLazyLog2; below that the weights 2^(s-M) stay < 2^8
                    // and every quantity remains exact to fp32 rounding.
                    bool grow = false;
#pragma unroll
                    for (int g = 0; g < G; ++g) grow |= fmaxf(sa[g], sb[g]) > M[g] + kLazyLog2;
                    float alpha[G];
                    bool rescale = (e != e_cur);
                    if (__any_sync(0xffffffffu, grow)) {
                        rescale = true;
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            const float m_new = fmaxf(M[g], redux_max_f32(fmaxf(sa[g], sb[g])));
                            alpha[g] = ex2_approx(M[g] - m_new);   // 0 while M is -inf
                            M[g] = m_new;
                        }
                    } else {
#pragma unroll
                        for (int g = 0; g < G; ++g) alpha[g] = 1.0f;
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float wa = va ? ex2_approx(sa[g] - M[g]) : 0.0f;
                        const float wb = vb ? ex2_approx(sb[g] - M[g]) : 0.0f;
                        Sl[g] = fmaf(Sl[g], alpha[g], wa + wb);
                        const float pa = wa * vsa * inv, pb = wb * vsb * inv;
                        const __half ha = __float2half_rn(pa), hb = __float2half_rn(pb);
                        p_hi[g * kPRowHalves + ta] = ha;
                        p_hi[g * kPRowHalves + tb] = hb;
                        p_lo[g * kPRowHalves + ta] = __float2half_rn(pa - __half2float(ha));
                        p_lo[g * kPRowHalves + tb] = __float2half_rn(pb - __half2float(hb));
                    }
                    if (rescale) {  // warp-uniform
                        const float two = __int_as_float((127 + max(-126, min(127, e_cur - e))) << 23);
                        float f0 = 0.0f, f1 = 0.0f;
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            if (g == col_head0) f0 = alpha[g] * two;
                            if (g == col_head1) f1 = alpha[g] * two;
                        }
#pragma unroll
                        for (int mt = 0; mt < 8; ++mt) {
                            acc[mt][0] *= f0; acc[mt][1] *= f1;
                            acc[mt][2] *= f0; acc[mt][3] *= f1;
                        }
                        e_cur = e;
                    }
                    __syncwarp();

                    // ---- segment 2c: acc += V . P on the tensor cores ----
                    // B columns: kPackPV, head n's high part (n < G) or head n - G's
                    // low part (G <= n < 2G); else the high part of head n in
                    // bh and its low part in bl (two MMAs)
                    uint32_t bh[8], bl[8];
                    const __half *rh = kPackPV ? (n < G ? p_hi + n * kPRowHalves
                                                        : (n < 2 * G ? p_lo + (n - G) * kPRowHalves : nullptr))
                                               : (n < G ? p_hi + n * kPRowHalves : nullptr);
                    if (rh) {
                        const int4 h0 = lds128(rh + t4 * 16);
                        const int4 h1 = lds128(rh + t4 * 16 + 8);
                        bh[0] = h0.x; bh[1] = h0.y; bh[2] = h0.z; bh[3] = h0.w;
                        bh[4] = h1.x; bh[5] = h1.y; bh[6] = h1.z; bh[7] = h1.w;
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) bh[i] = 0u;
                    }
                    if (!kPackPV && n < G) {
                        const int4 l0 = lds128(p_lo + n * kPRowHalves + t4 * 16);
                        const int4 l1 = lds128(p_lo + n * kPRowHalves + t4 * 16 + 8);
                        bl[0] = l0.x; bl[1] = l0.y; bl[2] = l0.z; bl[3] = l0.w;
                        bl[4] = l1.x; bl[5] = l1.y; bl[6] = l1.z; bl[7] = l1.w;
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) bl[i] = 0u;
                    }
                    // the stage's offset correction, one tile shared by all dims
                    float corr[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        mma_f16_16816(corr, kNegOffset, kNegOffset, kNegOffset, kNegOffset, bh[2 * s], bh[2 * s + 1]);
                        if (!kPackPV)
                            mma_f16_16816(corr, kNegOffset, kNegOffset, kNegOffset, kNegOffset, bl[2 * s], bl[2 * s + 1]);
                    }
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        const int d = mt * 16 + n;
                        const int4 v0 = lds128(vst + d * kStageTok + t4 * 16);
                        const int4 v1 = lds128(vst + (d + 8) * kStageTok + t4 * 16);
                        const uint32_t w0[4] = {(uint32_t)v0.x, (uint32_t)v0.y, (uint32_t)v0.z, (uint32_t)v0.w};
                        const uint32_t w1[4] = {(uint32_t)v1.x, (uint32_t)v1.y, (uint32_t)v1.z, (uint32_t)v1.w};
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            uint32_t a0, a2, a1, a3;
                            codes_to_sub2(w0[s], a0, a2);
                            codes_to_sub2(w1[s], a1, a3);
                            mma_f16_16816(acc[mt], a0, a1, a2, a3, bh[2 * s], bh[2 * s + 1]);
                            if (!kPackPV) mma_f16_16816(acc[mt], a0, a1, a2, a3, bl[2 * s], bl[2 * s + 1]);
                        }
                    }
                    // remove the stage's offset now, so that the accumulator never
                    // carries more than one stage of it (its rounding stays at the
                    // scale of the result)
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[mt][i] += corr[i];
                }
                __syncwarp();
                if (lane == 0) {
                    done[slot] = round + 1;
                    mbar_arrive(empty0 + 8 * slot);
                }
            }

            // ---- merge the 7 warp states of this segment into one record ----
            if (kPackPV) {
                // add the low parts' columns into the high parts' (the lanes
                // that hold columns 2*t4 < G, which the record write below reads)
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    if (G == 1) {
                        acc[mt][0] += acc[mt][1];
                        acc[mt][2] += acc[mt][3];
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[mt][i] += __shfl_xor_sync(0xffffffffu, acc[mt][i], G / 2);
                    }
                }
            }
            const float unit_scale = __int_as_float((127 + max(-126, min(127, e_cur))) << 23);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float s_w = warp_sum(Sl[g]);
                if (lane == 0) { red_m[g] = M[g]; red_s[g] = s_w; }
            }
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const int d0 = mt * 16 + n, h0 = 2 * t4, h1 = 2 * t4 + 1;
                if (h0 < G) {
                    red_acc[h0 * kHD + d0] = acc[mt][0] * kCodeUnit * unit_scale;
                    red_acc[h0 * kHD + d0 + 8] = acc[mt][2] * kCodeUnit * unit_scale;
                }
                if (h1 < G) {
                    red_acc[h1 * kHD + d0] = acc[mt][1] * kCodeUnit * unit_scale;
                    red_acc[h1 * kHD + d0 + 8] = acc[mt][3] * kCodeUnit * unit_scale;
                }
            }
            named_barrier_sync(1, kConsumerWarps * 32);
            const size_t rec = (size_t)c + u;
            // four dims per thread: one pass for G <= 4
            for (int idx = tid; idx < G * kHD / 4; idx += kConsumerWarps * 32) {
                const int g = idx / (kHD / 4), d = (idx % (kHD / 4)) * 4;
                float m = -INFINITY;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w)
                    m = fmaxf(m, reinterpret_cast<const float *>(smem + Lay::oScratch + w * Lay::kScratch)[G * kHD + g]);
                float s_sum = 0.0f;
                float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (m != -INFINITY) {
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) {
                        const float *r = reinterpret_cast<const float *>(smem + Lay::oScratch + w * Lay::kScratch);
                        const float f = ex2_approx(r[G * kHD + g] - m);
                        s_sum = fmaf(r[G * kHD + G + g], f, s_sum);
                        const float4 v = *reinterpret_cast<const float4 *>(r + g * kHD + d);
                        a.x = fmaf(v.x, f, a.x);
                        a.y = fmaf(v.y, f, a.y);
                        a.z = fmaf(v.z, f, a.z);
                        a.w = fmaf(v.w, f, a.w);
                    }
                }
                *reinterpret_cast<float4 *>(p.ws_acc + (rec * G + g) * kHD + d) = a;
                if (d == 0) {
                    p.ws_ml[(rec * G + g) * 2 + 0] = m;
                    p.ws_ml[(rec * G + g) * 2 + 1] = s_sum;
                }
            }
            if (tid == 0 && off == 0) p.ws_meta[u] = make_int2(c, meta_n);
            remaining -= seg_n;
            kbase += seg_n;
            off = 0;
            if (++h == p.nkv) { h = 0; ++b; }
        }
    }
    if (kMixed) pdl_wait();   // the 4-bit split's records are complete before this grid is
    pdl_launch_dependents();
    __syncthreads();
}

// Merge of the partial records of one (sequence, query head); thread = dim.
// [Day 9-2] §2 segment 3 generalised to several partial states:
// M = max_i M_i, S = sum_i S_i 2^(M_i - M), out = sum_i acc_i 2^(M_i - M) / S,
// the factors 2^(M_i - M) <= 1 by the approximate base-2 exponential, as the
// split kernel's weights, and the final division by the fast approximate one
// (S >= 1 and far below 2^126, where it is within 2 ulp; the library's exact
// exp2f and division cost this short kernel about 0.6 us of its critical
// path).  The records come from one split kernel,
// or from two (mixed precision by token age: the 4-bit split over [0, x) and
// the int8 split over [x, L)).
constexpr int kCombineRegs = 8;   // records merged from registers (more: the loop below)
constexpr int kCombineWide = 32;  // records of one source merged after one load round

__global__ void __launch_bounds__(kHD)
decode_combine_kernel(DecodeParams p, int G) {
    // The next kernel of the stream may be scheduled at once: every kernel of
    // this library waits for the grid before it to complete before it reads
    // what that grid writes (a decode step's split kernel, with the cache
    // declared ready, reads only the cache before that), and its CTAs take the
    // SMs that the split kernel before this one leaves.
    pdl_launch_dependents();
    pdl_wait();  // the split kernel's records are visible after this
    const int qh = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
    const int h = qh / G, g = qh % G;
    const int cap = p.max_blocks * kBS;
    const size_t u = (size_t)b * p.nkv + h;
    // the unit's record directories are loaded beside its length (one load
    // round); an entry is used only when the length says the unit has records
    // in that source (an empty unit's entry is not written by the split)
    const int2 meta0_raw = p.ws_meta[u];
    const int2 meta1_raw = p.ws_meta2 ? p.ws_meta2[u] : make_int2(0, 0);
    const int2 sp = seq_span(p, b, cap);
    float *o = p.out + ((size_t)b * p.nqh + qh) * kHD + d;
    if (sp.y == 0) { *o = 0.0f; return; }
    // source 0: this decode's records over [x, L); source 1: the 4-bit split's over [0, x)
    const bool has0 = sp.y > sp.x, has1 = p.ws_meta2 != nullptr && sp.x > 0;
    const int2 meta0 = has0 ? meta0_raw : make_int2(0, 0);
    const int2 meta1 = has1 ? meta1_raw : make_int2(0, 0);
    const size_t r00 = (size_t)meta0.x + u, r10 = (size_t)meta1.x + u;
    // the records of one source (both single-source paths below read these, so
    // that a call whose records all come from one split kernel gives the same
    // bits whichever source slot holds them)
    const bool one = meta0.y == 0 || meta1.y == 0;
    const float *ml1 = meta0.y ? p.ws_ml : p.ws_ml2, *acc1 = meta0.y ? p.ws_acc : p.ws_acc2;
    const size_t r01 = meta0.y ? r00 : r10;
    const int n1 = meta0.y ? meta0.y : meta1.y;
    if (one && n1 <= kCombineRegs) {
        // the usual case: every record's (M, S) and accumulator loaded at once,
        // then merged in the same order as below
        float mr[kCombineRegs], sr[kCombineRegs], ar[kCombineRegs];
#pragma unroll
        for (int j = 0; j < kCombineRegs; ++j) {
            if (j < n1) {
                const size_t r = (r01 + j) * G + g;
                const float2 ml = *reinterpret_cast<const float2 *>(ml1 + r * 2);
                mr[j] = ml.x;
                sr[j] = ml.y;
                ar[j] = acc1[r * kHD + d];
            }
        }
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < kCombineRegs; ++j)
            if (j < n1) m = fmaxf(m, mr[j]);
        float s_sum = 0.0f, a = 0.0f;
        if (m != -INFINITY) {
#pragma unroll
            for (int j = 0; j < kCombineRegs; ++j) {
                if (j < n1) {
                    const float f = ex2_approx(mr[j] - m);
                    s_sum = fmaf(sr[j], f, s_sum);
                    a = fmaf(ar[j], f, a);
                }
            }
        }
        *o = s_sum > 0.0f ? __fdividef(a, s_sum) : 0.0f;
        return;
    }
    if (one && n1 <= kCombineWide) {
        // up to 32 records of one source (a call of few long units): one load
        // round, then the same merge
        float2 mlr[kCombineWide];
        float ar[kCombineWide];
#pragma unroll
        for (int j = 0; j < kCombineWide; ++j) {
            if (j < n1) {
                const size_t r = (r01 + j) * G + g;
                mlr[j] = *reinterpret_cast<const float2 *>(ml1 + r * 2);
                ar[j] = acc1[r * kHD + d];
            }
        }
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < kCombineWide; ++j)
            if (j < n1) m = fmaxf(m, mlr[j].x);
        float s_sum = 0.0f, a = 0.0f;
        if (m != -INFINITY) {
#pragma unroll
            for (int j = 0; j < kCombineWide; ++j) {
                if (j < n1) {
                    const float f = ex2_approx(mlr[j].x - m);
                    s_sum = fmaf(mlr[j].y, f, s_sum);
                    a = fmaf(ar[j], f, a);
                }
            }
        }
        *o = s_sum > 0.0f ? __fdividef(a, s_sum) : 0.0f;
        return;
    }
    if (!one && meta0.y + meta1.y <= kCombineRegs) {
        // two sources, few records (a mixed-precision call of long units): both
        // sources' records loaded in one round (source 0's first), then merged
        float mr[kCombineRegs], sr[kCombineRegs], ar[kCombineRegs];
#pragma unroll
        for (int j = 0; j < kCombineRegs; ++j) {
            if (j < meta0.y + meta1.y) {
                const bool s0 = j < meta0.y;
                const size_t r = ((s0 ? r00 + j : r10 + (j - meta0.y))) * G + g;
                const float2 ml = *reinterpret_cast<const float2 *>((s0 ? p.ws_ml : p.ws_ml2) + r * 2);
                mr[j] = ml.x;
                sr[j] = ml.y;
                ar[j] = (s0 ? p.ws_acc : p.ws_acc2)[r * kHD + d];
            }
        }
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < kCombineRegs; ++j)
            if (j < meta0.y + meta1.y) m = fmaxf(m, mr[j]);
        float s_sum = 0.0f, a = 0.0f;
        if (m != -INFINITY) {
#pragma unroll
            for (int j = 0; j < kCombineRegs; ++j) {
                if (j < meta0.y + meta1.y) {
                    const float f = ex2_approx(mr[j] - m);
                    s_sum = fmaf(sr[j], f, s_sum);
                    a = fmaf(ar[j], f, a);
                }
            }
        }
        *o = s_sum > 0.0f ? __fdividef(a, s_sum) : 0.0f;
        return;
    }
    // more records: groups of kCombineRegs records, each group loaded at once
    // and merged into the running state with the same rescaling rule
    float m = -INFINITY, s_sum = 0.0f, a = 0.0f;
    auto merge_group = [&](const float *ml, const float *accp, size_t r0, int n) {
        float mr[kCombineRegs], sr[kCombineRegs], ar[kCombineRegs];
        float mg = -INFINITY;
#pragma unroll
        for (int j = 0; j < kCombineRegs; ++j) {
            if (j < n) {
                const size_t r = (r0 + j) * G + g;
                const float2 v = *reinterpret_cast<const float2 *>(ml + r * 2);
                mr[j] = v.x;
                sr[j] = v.y;
                ar[j] = accp[r * kHD + d];
                mg = fmaxf(mg, v.x);
            }
        }
        if (mg == -INFINITY) return;
        const float m_new = fmaxf(m, mg);
        const float f_old = ex2_approx(m - m_new);   // 0 while m is -inf
        s_sum *= f_old;
        a *= f_old;
#pragma unroll
        for (int j = 0; j < kCombineRegs; ++j) {
            if (j < n) {
                const float f = ex2_approx(mr[j] - m_new);
                s_sum = fmaf(sr[j], f, s_sum);
                a = fmaf(ar[j], f, a);
            }
        }
        m = m_new;
    };
    for (int j0 = 0; j0 < meta0.y; j0 += kCombineRegs)
        merge_group(p.ws_ml, p.ws_acc, r00 + j0, min(kCombineRegs, meta0.y - j0));
    for (int j0 = 0; j0 < meta1.y; j0 += kCombineRegs)
        merge_group(p.ws_ml2, p.ws_acc2, r10 + j0, min(kCombineRegs, meta1.y - j0));
    *o = s_sum > 0.0f ? __fdividef(a, s_sum) : 0.0f;
}

// The merge of the 4-bit decode, whose split writes unit u's records at
// u * nsplit + j: the records are loaded beside the unit's length (one load
// round, no record directory), and the length says how many of them this call
// wrote (int4_split_count); merged in the order of decode_combine_kernel.
__global__ void __launch_bounds__(kHD)
decode_combine_fixed_kernel(DecodeParams p, int G, int ns) {
    pdl_launch_dependents();   // as in decode_combine_kernel
    pdl_wait();
    const int qh = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
    const int h = qh / G, g = qh % G;
    const size_t u = (size_t)b * p.nkv + h;
    const int L = clamp_len(p.ctx_lens[b], p.max_blocks * kBS);
    float mr[kCombineRegs], sr[kCombineRegs], ar[kCombineRegs];
#pragma unroll
    for (int j = 0; j < kCombineRegs; ++j) {
        if (j < ns) {
            const size_t r = (u * ns + j) * G + g;
            const float2 ml = *reinterpret_cast<const float2 *>(p.ws_ml + r * 2);
            mr[j] = ml.x;
            sr[j] = ml.y;
            ar[j] = p.ws_acc[r * kHD + d];
        }
    }
    float *o = p.out + ((size_t)b * p.nqh + qh) * kHD + d;
    if (L == 0) { *o = 0.0f; return; }
    const int n1 = int4_split_count(L, ns);
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < kCombineRegs; ++j)
        if (j < n1) m = fmaxf(m, mr[j]);
    float s_sum = 0.0f, a = 0.0f;
    if (m != -INFINITY) {
#pragma unroll
        for (int j = 0; j < kCombineRegs; ++j) {
            if (j < n1) {
                const float f = ex2_approx(mr[j] - m);
                s_sum = fmaf(sr[j], f, s_sum);
                a = fmaf(ar[j], f, a);
            }
        }
    }
    *o = s_sum > 0.0f ? __fdividef(a, s_sum) : 0.0f;
}

int device_sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;
    }
    return cached[dev];
}

template <int G, bool kMixed, int kCtas>
cudaError_t launch_split_gm(const DecodeParams &p, cudaStream_t s) {
    using Lay = SplitLay<G, kMixed, kCtas>;
    static std::atomic<uint64_t> configured{0};
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(min(sms * kCtas, kMaxCtas));
    cfg.blockDim = dim3(kSplitThreads);
    cfg.dynamicSmemBytes = Lay::kBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return launch_after_setting(
        configured,
        [] {
            return cudaFuncSetAttribute(decode_split_kernel<G, kMixed, kCtas>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kBytes);
        },
        [&] { return cudaLaunchKernelEx(&cfg, decode_split_kernel<G, kMixed, kCtas>, p); });
}

template <int G>
cudaError_t launch_split_g(const DecodeParams &p, cudaStream_t s) {
    if (p.first_q8_block) {
        if constexpr (G == 2) return launch_split_gm<G, true, 2>(p, s);
        return launch_split_gm<G, true, 1>(p, s);
    }
    if constexpr (G == 2) {
        const int64_t units = (int64_t)p.batch * p.nkv;
        const int64_t stages_max = units * p.max_blocks * (kBS / kStageTok);
        const int sms = device_sm_count();
        if (units >= kTwoPerSmMinUnits && stages_max >= (int64_t)kTwoPerSmMinStages * 2 * sms)
            return launch_split_gm<G, false, 2>(p, s);
    }
    return launch_split_gm<G, false, 1>(p, s);
}

}  // namespace

bool make_decode_plan(int batch, int nqh, int nkv, int max_blocks, DecodePlan *plan) {
    if (batch < 0 || nqh <= 0 || nkv <= 0 || max_blocks <= 0 || nqh % nkv) return false;
    const int G = nqh / nkv;
    auto align = [](size_t x) { return (x + 255) & ~(size_t)255; };
    plan->group = G;
    plan->units = (int64_t)batch * nkv;
    plan->records = kMaxCtas + plan->units;
    plan->meta_offset = 0;
    plan->ml_offset = align((size_t)plan->units * sizeof(int2));
    plan->acc_offset = plan->ml_offset + align((size_t)plan->records * G * 2 * sizeof(float));
    plan->bytes = plan->acc_offset + align((size_t)plan->records * G * kHD * sizeof(float));
    return true;
}

cudaError_t launch_decode_split(const DecodeParams &p, int group, cudaStream_t s) {
    switch (group) {
        case 1: return launch_split_g<1>(p, s);
        case 2: return launch_split_g<2>(p, s);
        case 4: return launch_split_g<4>(p, s);
        case 8: return launch_split_g<8>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode_combine_fixed(const DecodeParams &p, int group, int nsplit, cudaStream_t s) {
    if (nsplit < 1 || nsplit > kCombineRegs) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.nqh, p.batch);
    cfg.blockDim = dim3(kHD);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_combine_fixed_kernel, p, group, nsplit);
}

cudaError_t launch_decode_combine(const DecodeParams &p, int group, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.nqh, p.batch);
    cfg.blockDim = dim3(kHD);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel, p, group);
}

}  // namespace kvq8
