/*
 * CPU oracle for exact QSA block selection -- TEST INFRASTRUCTURE ONLY.
 * Declarations for qsa_oracle.c; nothing outside the tests, the smoke check
 * and the benchmark's CPU-baseline leg includes or links this.
 *
 * Layouts (all row-major, host memory owned by the caller):
 *   q       float  [nq][4][128]
 *   kblk    float  [>= active][128]
 *   kq8     int8   [>= active][128], kscale uint16 (IEEE binary16) [>= active]
 *   S       double [nq][active]      (scores, written)
 *   scores  float  [nq][active]      (given fp32 scores, read)
 *   ids     int32  [nq][k]           (written: ascending ids, -1 padding)
 *   attention: kq, vq int8 [ncells][128], ks, vs uint16 (binary16) [ncells],
 *              ids int32 [nq][k] (read), out double [nq][4][128] (written)
 *   summary:   key float [b1-b0][128], kq8 int8 [b1-b0][128], kscale uint16 [b1-b0]
 *              (rows of blocks b0..b1-1, written; key or kq8+kscale may be NULL)
 * nthreads <= 0 uses every online core.
 */
#ifndef QSA_ORACLE_H
#define QSA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int qsa_oracle_default_threads(void);
double qsa_oracle_half_to_double(uint16_t h);
void qsa_oracle_scores(const float *q, const float *kblk, long nq, long active,
                       double *S, int nthreads);
void qsa_oracle_scores_q8(const float *q, const int8_t *kq8, const uint16_t *kscale,
                          long nq, long active, double *S, int nthreads);
void qsa_oracle_topk_f64(const double *S, long nq, long active, long k, int32_t *ids,
                         int nthreads);
void qsa_oracle_topk_f32(const float *scores, long nq, long active, long k, int32_t *ids,
                         int nthreads);
uint16_t qsa_oracle_float_to_half(float f);
void qsa_oracle_block_summary(const int8_t *kq, const uint16_t *ks, long ncells, long b0, long b1,
                              float *key, int8_t *kq8, uint16_t *kscale);
void qsa_oracle_sparse_attn(const float *q, const int8_t *kq, const uint16_t *ks, const int8_t *vq,
                            const uint16_t *vs, long ncells, const int32_t *ids, long nq, long k,
                            double *out, int nthreads);

#ifdef __cplusplus
}
#endif

#endif
