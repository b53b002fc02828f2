/*
 * kvq8_oracle.c -- plain CPU oracle for INT8-KV decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg use it.  It shares no header, helper or constant with the
 * CUDA library: every rule below is restated here from the pages.
 *
 * Pages (web articles of the "0.8MB 跑通 Qwen" tutorial series and one blog):
 *   [Day 9-1] "推理引擎的 KV 也量化——q8 KV 把缓存与 decode 带宽压到一半"
 *   [Day 9-2] "flash_attn_single_q_q8_neon——单 q 单遍扫全 KV"
 *   [Day 9-3] "q8 KV 精度对照——量化进注意力，输出差多少"
 *   [UltraQuant] the UltraQuant 4-bit KV-cache blog (AMD RX 7900 XTX)
 *
 * Precision: every quantisation step is done in IEEE fp32, exactly as the
 * engine on the pages does it (its code is fp32 C), because those steps
 * decide integer codes.  Float->int rounding is round-half-to-even
 * (nearbyintf under the default rounding mode) -- the pages say "round"
 * without naming a tie rule; half-even is the reading taken, and ties have
 * measure zero on random data.  Everything after the integer dot products
 * (score scaling, softmax, weighted sum) is accumulated in fp64.
 *
 * Build with -O2 -fno-fast-math -ffp-contract=off so that no multiply-add is
 * fused and no IEEE rule is relaxed.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "kvq8_oracle.h"

/* ------------------------------------------------------------------------ */
/* Non-finite inputs.  The pages state every rule for finite values only.   */
/* Reading taken: a unit of quantisation (a K/V row, a query 32-block, an   */
/* INT4 group) that holds a NaN or an infinity is quantised exactly as if   */
/* all of its values were zero; each quantiser returns how many units it    */
/* replaced so.  With finite input every float->int conversion below sees a */
/* finite value inside the int range.                                       */
/* ------------------------------------------------------------------------ */
static int all_finite(const float *x, int n)
{
    for (int i = 0; i < n; ++i)
        if (!isfinite(x[i]))
            return 0;
    return 1;
}

/* ------------------------------------------------------------------------ */
/* K/V write path: per-(token, head) max-abs INT8 quantisation.             */
/* [Day 9-3] §2 (quantisation rule taken from the engine's write path):     */
/* over the hd values of one (token, head) row take max_abs, scale =       */
/* max_abs/127, q = round(v/scale) clamped to [-127, 127], one fp32 scale   */
/* per row; [Day 9-1] §2 (kv_quantize_per_head call, one scale per token    */
/* per head).  An all-zero row (pages silent) gets scale 0 and codes 0; so  */
/* does a row holding a NaN or an infinity (counted in the return value).   */
/* ------------------------------------------------------------------------ */
int64_t orc_kv_quantize_rows(const float *x, int64_t n_rows, int hd,
                             int8_t *q, float *scale)
{
    int64_t replaced = 0;
    for (int64_t r = 0; r < n_rows; ++r) {
        const float *v = x + r * (int64_t)hd;
        int8_t *qr = q + r * (int64_t)hd;
        if (!all_finite(v, hd)) {
            /* the row of zeros: max_abs 0, scale 0, every code 0 */
            ++replaced;
            scale[r] = 0.0f;
            memset(qr, 0, (size_t)hd);
            continue;
        }
        float max_abs = 0.0f;
        for (int i = 0; i < hd; ++i) {
            float a = fabsf(v[i]);
            if (a > max_abs)
                max_abs = a;
        }
        float s = max_abs / 127.0f;
        scale[r] = s;
        for (int i = 0; i < hd; ++i) {
            float c = 0.0f;
            if (s != 0.0f) {
                float t = v[i] / s;
                c = nearbyintf(t);
                if (c > 127.0f)
                    c = 127.0f;
                if (c < -127.0f)
                    c = -127.0f;
            }
            qr[i] = (int8_t)(int)c;
        }
    }
    return replaced;
}

/* Dequantisation v = q * scale ([Day 9-3] §2, the inverse of the rule above),
 * in fp32 as the engine stores and uses it. */
void orc_kv_dequantize_rows(const int8_t *q, const float *scale,
                            int64_t n_rows, int hd, float *out)
{
    for (int64_t r = 0; r < n_rows; ++r)
        for (int i = 0; i < hd; ++i)
            out[r * (int64_t)hd + i] = (float)q[r * (int64_t)hd + i] * scale[r];
}

/* ------------------------------------------------------------------------ */
/* Q quantisation in 32-element blocks ("Q8_0 isomorphic").                 */
/* [Day 9-2] §2 segment 1: per block qm = max|x|; if qm < 1e-6 then qm = 1; */
/* block scale = qm * (1/127); iq = 127/qm; code = clamp(x*iq, -128, 127).  */
/* The page's conversion to int8 is garbled; round-half-even is the reading */
/* taken (same rule as K/V).  n must be a multiple of 32.  A block holding  */
/* a NaN or an infinity is quantised as a block of zeros (qm 0 -> 1, scale  */
/* 1/127, codes 0); the return value counts such blocks.                    */
/* ------------------------------------------------------------------------ */
int64_t orc_q_quantize_blocks(const float *x, int64_t n, int8_t *qi, float *qsc)
{
    const float kvq_inv = 1.0f / 127.0f;
    static const float zeros[32];
    int64_t replaced = 0;
    for (int64_t b = 0; b < n / 32; ++b) {
        const float *xb = x + b * 32;
        if (!all_finite(xb, 32)) {
            ++replaced;
            xb = zeros;
        }
        float qm = 0.0f;
        for (int i = 0; i < 32; ++i)
            qm = fmaxf(qm, fabsf(xb[i]));
        if (qm < 1e-6f)
            qm = 1.0f;
        qsc[b] = qm * kvq_inv;
        float iq = 127.0f / qm;
        for (int i = 0; i < 32; ++i) {
            float t = xb[i] * iq;
            float c = nearbyintf(t);
            if (c > 127.0f)
                c = 127.0f;
            if (c < -128.0f)
                c = -128.0f;
            qi[b * 32 + i] = (int8_t)(int)c;
        }
    }
    return replaced;
}

/* ------------------------------------------------------------------------ */
/* Scores of one quantised query against L quantised key rows.              */
/* [Day 9-2] §2 segment 2 and its "three key points": per 32-block an       */
/* integer dot of the int8 codes; the float value is rebuilt by multiplying */
/* each block dot by the query block scale, summing over blocks, then       */
/* multiplying by the key row scale and the softmax scale 1/sqrt(hd).       */
/* The block dots are exact integers; the rest is fp64.                     */
/* ------------------------------------------------------------------------ */
static void scores_q8(const int8_t *qi, const float *qsc, int hd,
                      const int8_t *kq, const float *ks, int64_t L,
                      double sm_scale, double *s)
{
    int nblk = hd / 32;
    for (int64_t t = 0; t < L; ++t) {
        const int8_t *kt = kq + t * (int64_t)hd;
        double acc = 0.0;
        for (int b = 0; b < nblk; ++b) {
            int32_t dot = 0;
            for (int i = b * 32; i < b * 32 + 32; ++i)
                dot += (int32_t)qi[i] * (int32_t)kt[i];
            acc += (double)dot * (double)qsc[b];
        }
        s[t] = acc * (double)ks[t] * sm_scale;
    }
}

void orc_scores_q8(const int8_t *qi, const float *qsc, int hd,
                   const int8_t *kq, const float *ks, int64_t L,
                   float sm_scale, double *s)
{
    scores_q8(qi, qsc, hd, kq, ks, L, (double)sm_scale, s);
}

/* ------------------------------------------------------------------------ */
/* Decode attention, three-pass form ("textbook" form the pages contrast    */
/* with the single pass): scores -> max-subtracted softmax -> weighted sum  */
/* of dequantised V.  [Day 9-3] §1-§2 (score = Q.K^T/sqrt(128), subtract    */
/* max, stable softmax, weighted V); [Day 9-2] §1 and §3 (the three-pass    */
/* form is functionally equal to the single pass).                          */
/* One query head; K/V rows of its kv head are contiguous [L][hd].          */
/* weights (nullable) receives the L normalised softmax weights.            */
/* L == 0 (pages silent) gives out = 0.                                     */
/* Returns 0, or -1 when scratch memory cannot be had.                      */
/* ------------------------------------------------------------------------ */
int orc_decode_q8_three_pass(const int8_t *qi, const float *qsc, int hd,
                             const int8_t *kq, const float *ks,
                             const int8_t *vq, const float *vs, int64_t L,
                             float sm_scale, double *out, double *weights)
{
    for (int i = 0; i < hd; ++i)
        out[i] = 0.0;
    if (L <= 0)
        return 0;
    double *s = (double *)malloc((size_t)L * sizeof(double));
    if (!s)
        return -1;
    /* pass 1: scores */
    scores_q8(qi, qsc, hd, kq, ks, L, (double)sm_scale, s);
    double mu = s[0];
    for (int64_t t = 1; t < L; ++t)
        if (s[t] > mu)
            mu = s[t];
    /* pass 2: exponentials and their sum */
    double S = 0.0;
    for (int64_t t = 0; t < L; ++t) {
        s[t] = exp(s[t] - mu);
        S += s[t];
    }
    /* pass 3: weighted sum of dequantised V */
    for (int64_t t = 0; t < L; ++t) {
        double w = s[t] / S;
        if (weights)
            weights[t] = w;
        const int8_t *vt = vq + t * (int64_t)hd;
        for (int i = 0; i < hd; ++i)
            out[i] += w * ((double)vt[i] * (double)vs[t]);
    }
    free(s);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Decode attention, single-pass online form, in fp64.                      */
/* [Day 9-2] §1 and §2 segments 2-3: running max M (starts at -1e9) and     */
/* running exp-sum S; a score above M rescales S and the V accumulator by   */
/* exp(M_old - s) and becomes the new M with weight 1, otherwise its weight */
/* is exp(s - M); the accumulator gathers int8 V times (weight * v_scale);  */
/* one division by S at the end.  Used only to pin the three-pass form.     */
/* ------------------------------------------------------------------------ */
int orc_decode_q8_online(const int8_t *qi, const float *qsc, int hd,
                         const int8_t *kq, const float *ks,
                         const int8_t *vq, const float *vs, int64_t L,
                         float sm_scale, double *out)
{
    for (int i = 0; i < hd; ++i)
        out[i] = 0.0;
    if (L <= 0)
        return 0;
    double *acc = (double *)calloc((size_t)hd, sizeof(double));
    if (!acc)
        return -1;
    double M = -1e9, S = 0.0;
    for (int64_t t = 0; t < L; ++t) {
        double s;
        scores_q8(qi, qsc, hd, kq + t * (int64_t)hd, ks + t, 1,
                  (double)sm_scale, &s);
        double w;
        if (s > M) {
            double c = exp(M - s);
            S *= c;
            for (int i = 0; i < hd; ++i)
                acc[i] *= c;
            M = s;
            w = 1.0;
        } else {
            w = exp(s - M);
        }
        S += w;
        const int8_t *vt = vq + t * (int64_t)hd;
        double wv = w * (double)vs[t];
        for (int i = 0; i < hd; ++i)
            acc[i] += (double)vt[i] * wv;
    }
    for (int i = 0; i < hd; ++i)
        out[i] = acc[i] / S;
    free(acc);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Plain softmax attention of one float query over float K/V rows, fp64.    */
/* The fp32-KV baseline of [Day 9-3] §1 (Q.K^T -> stable softmax ->         */
/* weighted V, nothing quantised) and, fed dequantised K/V, its q8-KV arm.  */
/* Also the attention of the 4-bit path, which takes a float query against  */
/* dequantised K/V ([UltraQuant] §4.1 / §5.3: dequantise, then standard     */
/* attention).  L == 0 gives out = 0.                                       */
/* ------------------------------------------------------------------------ */
int orc_attention_f64(const float *q, const float *k, const float *v,
                      int64_t L, int hd, float sm_scale, double *out)
{
    for (int i = 0; i < hd; ++i)
        out[i] = 0.0;
    if (L <= 0)
        return 0;
    double *s = (double *)malloc((size_t)L * sizeof(double));
    if (!s)
        return -1;
    for (int64_t t = 0; t < L; ++t) {
        double d = 0.0;
        for (int i = 0; i < hd; ++i)
            d += (double)q[i] * (double)k[t * (int64_t)hd + i];
        s[t] = d * (double)sm_scale;
    }
    double mu = s[0];
    for (int64_t t = 1; t < L; ++t)
        if (s[t] > mu)
            mu = s[t];
    double S = 0.0;
    for (int64_t t = 0; t < L; ++t) {
        s[t] = exp(s[t] - mu);
        S += s[t];
    }
    for (int64_t t = 0; t < L; ++t) {
        double w = s[t] / S;
        for (int i = 0; i < hd; ++i)
            out[i] += w * (double)v[t * (int64_t)hd + i];
    }
    free(s);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Asymmetric INT4 group quantisation with nibble packing.                  */
/* [UltraQuant] §3.2 code: per group of `group` consecutive values,         */
/* scale = (max - min)/15 (1.0 when max == min), zero = round(-min/scale),  */
/* q = clamp(round(x/scale + zero), 0, 15); two codes per byte, the even    */
/* element in the high nibble.  Dequantise (q - zero) * scale.              */
/* torch.round is round-half-even, so nearbyintf is the same rule.  scale   */
/* and zero stay fp32 (the page keeps them in float tensors).               */
/* n must be a multiple of group, group even (at most 1024).  A group that  */
/* holds a NaN or an infinity is quantised as a group of zeros (scale 1,    */
/* zero = round(-0/1) = -0, codes 0); the return value counts such groups.  */
/* ------------------------------------------------------------------------ */
int64_t orc_int4_quantize_groups(const float *x, int64_t n, int group,
                                 uint8_t *packed, float *scale, float *zero)
{
    static const float zeros[1024];
    int64_t ng = n / group;
    int64_t replaced = 0;
    if (group > 1024)
        return -1;
    for (int64_t g = 0; g < ng; ++g) {
        const float *xg = x + g * group;
        if (!all_finite(xg, group)) {
            ++replaced;
            xg = zeros;
        }
        float mx = xg[0], mn = xg[0];
        for (int i = 1; i < group; ++i) {
            if (xg[i] > mx)
                mx = xg[i];
            if (xg[i] < mn)
                mn = xg[i];
        }
        float s = (mx != mn) ? (mx - mn) / 15.0f : 1.0f;
        float z = nearbyintf(-mn / s);
        scale[g] = s;
        zero[g] = z;
        for (int i = 0; i < group; i += 2) {
            int c[2];
            for (int j = 0; j < 2; ++j) {
                float t = xg[i + j] / s + z;
                float r = nearbyintf(t);
                if (r < 0.0f)
                    r = 0.0f;
                if (r > 15.0f)
                    r = 15.0f;
                c[j] = (int)r;
            }
            packed[(g * group + i) / 2] = (uint8_t)((c[0] << 4) | c[1]);
        }
    }
    return replaced;
}

void orc_int4_dequantize_groups(const uint8_t *packed, const float *scale,
                                const float *zero, int64_t n, int group,
                                float *out)
{
    for (int64_t e = 0; e < n; ++e) {
        uint8_t byte = packed[e / 2];
        int c = (e % 2 == 0) ? (byte >> 4) : (byte & 0x0F);
        int64_t g = e / group;
        out[e] = ((float)c - zero[g]) * scale[g];
    }
}

/*
 * Mixed precision by token age ([UltraQuant] §3.3, "practical note": tokens in
 * time blocks share one precision; recent blocks stay 8-bit, the oldest are
 * requantised to 4-bit).  One query head against a context whose first n4
 * tokens are 4-bit (given here as their dequantised fp32 rows k4, v4) and
 * whose remaining L8 tokens are int8 (codes and per-row scales).  Scores: the
 * fp32 query against k4 for the old tokens ([UltraQuant] §4.1: dequantise,
 * then standard attention); the [Day 9-2] integer block dots for the recent
 * ones.  Then the same three passes as orc_decode_q8_three_pass over the
 * concatenated sequence (old first), all in fp64.
 */
int orc_decode_mixed(const float *q, const int8_t *qi, const float *qsc, int hd,
                     const float *k4, const float *v4, int64_t n4,
                     const int8_t *kq, const float *ks, const int8_t *vq, const float *vs,
                     int64_t L8, float sm_scale, double *out)
{
    for (int i = 0; i < hd; ++i)
        out[i] = 0.0;
    const int64_t L = n4 + L8;
    if (L <= 0)
        return 0;
    double *s = (double *)malloc((size_t)L * sizeof(double));
    if (!s)
        return -1;
    /* pass 1: scores */
    for (int64_t t = 0; t < n4; ++t) {
        double d = 0.0;
        for (int i = 0; i < hd; ++i)
            d += (double)q[i] * (double)k4[t * (int64_t)hd + i];
        s[t] = d * (double)sm_scale;
    }
    if (L8 > 0)
        scores_q8(qi, qsc, hd, kq, ks, L8, (double)sm_scale, s + n4);
    double mu = s[0];
    for (int64_t t = 1; t < L; ++t)
        if (s[t] > mu)
            mu = s[t];
    /* pass 2: exponentials and their sum */
    double S = 0.0;
    for (int64_t t = 0; t < L; ++t) {
        s[t] = exp(s[t] - mu);
        S += s[t];
    }
    /* pass 3: weighted sum of the dequantised V rows */
    for (int64_t t = 0; t < n4; ++t) {
        const double w = s[t] / S;
        for (int i = 0; i < hd; ++i)
            out[i] += w * (double)v4[t * (int64_t)hd + i];
    }
    for (int64_t t = 0; t < L8; ++t) {
        const double w = s[n4 + t] / S;
        const int8_t *vt = vq + t * (int64_t)hd;
        for (int i = 0; i < hd; ++i)
            out[i] += w * ((double)vt[i] * (double)vs[t]);
    }
    free(s);
    return 0;
}

int orc_version(void) { return 1; }
