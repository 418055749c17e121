/*
 * oracle.h -- the CPU oracle's own declarations (test infrastructure only; see
 * oracle.c).  Deliberately independent of the CUDA library's header: the config
 * struct below is this file's own definition of the same fields.
 */
#ifndef ORACLE_H
#define ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_Q8 = 2 };
enum { ORC_Q8_BLOCK = 32 };
enum {
    ORC_OK = 0,
    ORC_EINVAL = -1,
    ORC_ENOMEM = -2,
    ORC_ECAPACITY = -3,
    ORC_EPOS = -4,
    ORC_ESTATE = -5
};

typedef struct {
    int32_t dim, n_layers, n_heads, n_kv_heads, head_dim, hidden, vocab, max_seq, max_batch;
    float rope_theta, norm_eps;
    int32_t weight_dtype, kv_dtype;
} orc_config;

typedef struct orc_model orc_model;

/* scalar pieces, exported so the tests can pin each one on its own */
float orc_bf16_up(uint16_t b);
float orc_bf16_round(float f);
void orc_rmsnorm(float *out, const float *x, const float *g, int n, float eps);
void orc_matvec(float *out, const float *w, const float *x, int n_in, int n_out);
void orc_rope(float *v, int n_heads, int head_dim, int pos, float theta);
void orc_attend(float *out, const float *q, const float *kc, const float *vc, int n_ctx,
                int head_dim, float *scores);
void orc_silu_mul(float *h, const float *a, const float *b, int n);
int32_t orc_argmax(const float *x, int n);
void orc_quantize_q8_row(const float *w, int n, int8_t *q, float *d);

/* the model */
size_t orc_weight_count(const orc_config *c);
int orc_create(const orc_config *cfg, const void *weights, size_t nbytes, orc_model **out);
void orc_destroy(orc_model *m);
int orc_prefill(orc_model *m, int32_t seq, const int32_t *tokens, int32_t n, float *last_logits,
                int32_t *next_id);
int orc_decode_step(orc_model *m, int32_t batch, const int32_t *seq_ids, const int32_t *tokens,
                    const int32_t *positions, float *logits, int32_t *next_ids);
int orc_reset(orc_model *m, int32_t seq);
int32_t orc_seq_len(const orc_model *m, int32_t seq);
int64_t orc_passes(const orc_model *m);
int orc_copy_kv(const orc_model *m, int32_t layer, int32_t seq, float *k_out, float *v_out);
int orc_layer0_kv(const orc_model *m, int32_t tok, int32_t pos, float *k_out, float *v_out);
int orc_forward_uncached(orc_model *m, const int32_t *tokens, int32_t n, float *last_logits,
                         int32_t *next_id);

#ifdef __cplusplus
}
#endif
#endif
