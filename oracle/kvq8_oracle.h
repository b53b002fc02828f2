/*
 * kvq8_oracle.h -- declarations of the CPU oracle (test infrastructure only;
 * see kvq8_oracle.c for the rules each function restates and their sources).
 * This header is private to oracle/: the CUDA library never includes it.
 */
#ifndef KVQ8_ORACLE_H
#define KVQ8_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int64_t orc_kv_quantize_rows(const float *x, int64_t n_rows, int hd,
                             int8_t *q, float *scale);
void orc_kv_dequantize_rows(const int8_t *q, const float *scale,
                            int64_t n_rows, int hd, float *out);
int64_t orc_q_quantize_blocks(const float *x, int64_t n, int8_t *qi, float *qsc);
void orc_scores_q8(const int8_t *qi, const float *qsc, int hd,
                   const int8_t *kq, const float *ks, int64_t L,
                   float sm_scale, double *s);
int orc_decode_q8_three_pass(const int8_t *qi, const float *qsc, int hd,
                             const int8_t *kq, const float *ks,
                             const int8_t *vq, const float *vs, int64_t L,
                             float sm_scale, double *out, double *weights);
int orc_decode_q8_online(const int8_t *qi, const float *qsc, int hd,
                         const int8_t *kq, const float *ks,
                         const int8_t *vq, const float *vs, int64_t L,
                         float sm_scale, double *out);
int orc_attention_f64(const float *q, const float *k, const float *v,
                      int64_t L, int hd, float sm_scale, double *out);
int64_t orc_int4_quantize_groups(const float *x, int64_t n, int group,
                                 uint8_t *packed, float *scale, float *zero);
void orc_int4_dequantize_groups(const uint8_t *packed, const float *scale,
                                const float *zero, int64_t n, int group,
                                float *out);
int orc_decode_mixed(const float *q, const int8_t *qi, const float *qsc, int hd,
                     const float *k4, const float *v4, int64_t n4,
                     const int8_t *kq, const float *ks, const int8_t *vq, const float *vs,
                     int64_t L8, float sm_scale, double *out);
int orc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ8_ORACLE_H */
