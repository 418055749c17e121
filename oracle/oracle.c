/*
 * oracle.c -- plain, slow, single-threaded fp32 CPU oracle of the KV-cached greedy
 * decode step of a LLaMA-style decoder.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this
 * file: only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header, table or constant with the CUDA library; the two meet
 * only at the seeded inputs made by the `synth` module.
 *
 * What it computes (all in fp32, every sum in ascending index order, no FMA
 * contraction -- build with -ffp-contract=off):
 *
 *   kasahare 0.4.0 (simple-llm), "Architecture": per block
 *       xn   = attn_norm(x)
 *       q,k,v = Wq xn, Wk xn, Wv xn                      (no biases)
 *       q,k  = RoPE(q, k, pos)
 *       attn = softmax(q . K^T / sqrt(d_head)) . V        (GQA, all cached positions)
 *       x    = x + Wo attn                                (residual)
 *       xn   = ffn_norm(x)
 *       x    = x + W2( silu(W1 xn) * (W3 xn) )            (SwiGLU, residual)
 *   The printed equations overwrite the residual stream with its normalised copy;
 *   the only reading consistent with their "# residual" comments is the standard
 *   pre-norm block above, where the residual is the un-normalised stream.
 *   Final: logits = E . rmsnorm(x, output_norm) with the tied embedding E
 *   (kasahare, "Optimisations": tied input/output embeddings), then greedy argmax.
 *
 *   GOTOken: An Inference Engine in QBasic, "About one token per second": every
 *   projection is  xout(i) = sum_j W(i, j) x(j)  with W row-major and a single fp32
 *   accumulator starting at zero; "Loading the model and tokenizer": a bf16 weight
 *   widens to fp32 by shifting its 16 bits left by 16.  The KV cache keeps the key and
 *   value rows of position t, which depend only on tokens 0..t, and reuses them; the
 *   cached run is bit-identical to the uncached one.
 *
 * Readings where the pages are silent (each is listed with its reason in the design
 * notes): RMSNorm eps comes from the config (1e-5); RoPE rotates the half-split pairs
 * (i, i + hd/2) with frequency theta^(-2i/hd), angle and sin/cos taken in double and
 * rounded to fp32; query head h reads kv head h / (H/KV); softmax subtracts the max,
 * exponentiates with expf, divides by the ascending sum, then weights V; argmax takes
 * the lowest index on a tie; a bf16 KV cache rounds k and v to nearest-even on append.
 *
 * Block-quantised int8 weights (kasahare 0.4.0, "Where to go from here": INT8 weight
 * loading, block-quantised like GGUF; the pages give no format, so this is the plainest
 * one): every row of every projection matrix and of the tied embedding is cut into
 * blocks of ORC_Q8_BLOCK consecutive elements (the last block of a row may be shorter);
 * a block keeps d = max|w| / 127 and q_i = w_i / d rounded to the nearest integer, halves
 * away from zero (an all-zero block: d = 0, q = 0).  The weight the model then uses is
 * the fp32 product d * q_i; nothing else changes.  The norm gains stay fp32.
 */
#include "oracle.h"

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- scalar pieces */

float orc_bf16_up(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

float orc_bf16_round(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u) {
        /* inf stays inf; a NaN stays a (quiet) NaN */
        if (u & 0x007fffffu) u |= 0x00400000u;
        u &= 0xffff0000u;
    } else {
        u += 0x7fffu + ((u >> 16) & 1u);
        u &= 0xffff0000u;
    }
    memcpy(&f, &u, sizeof f);
    return f;
}

void orc_rmsnorm(float *out, const float *x, const float *g, int n, float eps) {
    float ss = 0.0f;
    for (int i = 0; i < n; i++) ss = ss + x[i] * x[i];
    float ms = ss / (float)n;
    float r = 1.0f / sqrtf(ms + eps);
    for (int i = 0; i < n; i++) out[i] = (x[i] * r) * g[i];
}

void orc_matvec(float *out, const float *w, const float *x, int n_in, int n_out) {
    for (int i = 0; i < n_out; i++) {
        const float *row = w + (size_t)i * (size_t)n_in;
        float acc = 0.0f;
        for (int j = 0; j < n_in; j++) acc = acc + row[j] * x[j];
        out[i] = acc;
    }
}

void orc_rope(float *v, int n_heads, int head_dim, int pos, float theta) {
    int half = head_dim / 2;
    for (int h = 0; h < n_heads; h++) {
        float *u = v + (size_t)h * head_dim;
        for (int i = 0; i < half; i++) {
            double freq = pow((double)theta, -2.0 * (double)i / (double)head_dim);
            double ang = (double)pos * freq;
            float c = (float)cos(ang);
            float s = (float)sin(ang);
            float a = u[i];
            float b = u[i + half];
            u[i] = a * c - b * s;
            u[i + half] = a * s + b * c;
        }
    }
}

void orc_attend(float *out, const float *q, const float *kc, const float *vc, int n_ctx,
                int head_dim, float *scores) {
    float scale = 1.0f / sqrtf((float)head_dim);
    for (int t = 0; t < n_ctx; t++) {
        const float *k = kc + (size_t)t * head_dim;
        float acc = 0.0f;
        for (int i = 0; i < head_dim; i++) acc = acc + q[i] * k[i];
        scores[t] = acc * scale;
    }
    float m = scores[0];
    for (int t = 1; t < n_ctx; t++)
        if (scores[t] > m) m = scores[t];
    float z = 0.0f;
    for (int t = 0; t < n_ctx; t++) {
        scores[t] = expf(scores[t] - m);
        z = z + scores[t];
    }
    for (int t = 0; t < n_ctx; t++) scores[t] = scores[t] / z;
    for (int i = 0; i < head_dim; i++) out[i] = 0.0f;
    for (int t = 0; t < n_ctx; t++) {
        const float *v = vc + (size_t)t * head_dim;
        for (int i = 0; i < head_dim; i++) out[i] = out[i] + scores[t] * v[i];
    }
}

void orc_silu_mul(float *h, const float *a, const float *b, int n) {
    for (int i = 0; i < n; i++) h[i] = (a[i] / (1.0f + expf(-a[i]))) * b[i];
}

/* one row of n weights to int8 blocks of ORC_Q8_BLOCK: q[n], d[ceil(n / ORC_Q8_BLOCK)] */
void orc_quantize_q8_row(const float *w, int n, int8_t *q, float *d) {
    for (int b0 = 0, blk = 0; b0 < n; b0 += ORC_Q8_BLOCK, blk++) {
        int b1 = b0 + ORC_Q8_BLOCK < n ? b0 + ORC_Q8_BLOCK : n;
        float amax = 0.0f;
        for (int i = b0; i < b1; i++) {
            float a = fabsf(w[i]);
            if (a > amax) amax = a;
        }
        float s = amax / 127.0f;
        d[blk] = s;
        for (int i = b0; i < b1; i++) {
            float v = s > 0.0f ? roundf(w[i] / s) : 0.0f;
            if (v > 127.0f) v = 127.0f;
            if (v < -127.0f) v = -127.0f;
            q[i] = (int8_t)v;
        }
    }
}

/* replace each of `rows` rows of n weights by its block-quantised value d * q */
static int q8_dequantize_rows(float *w, size_t rows, int n) {
    int8_t *q = malloc((size_t)n);
    float *d = malloc(((size_t)n / ORC_Q8_BLOCK + 1) * sizeof(float));
    if (!q || !d) {
        free(q);
        free(d);
        return ORC_ENOMEM;
    }
    for (size_t r = 0; r < rows; r++) {
        float *row = w + r * (size_t)n;
        orc_quantize_q8_row(row, n, q, d);
        for (int i = 0; i < n; i++) row[i] = d[i / ORC_Q8_BLOCK] * (float)q[i];
    }
    free(q);
    free(d);
    return ORC_OK;
}

int32_t orc_argmax(const float *x, int n) {
    int32_t best = 0;
    for (int i = 0; i < n; i++)
        if (isnan(x[i])) return -1;
    for (int i = 1; i < n; i++)
        if (x[i] > x[best]) best = i;
    return best;
}

/* ---------------------------------------------------------------- the model */

typedef struct {
    const float *attn_norm, *wq, *wk, *wv, *wo, *ffn_norm, *w1, *w3, *w2;
} orc_layer;

struct orc_model {
    orc_config c;
    float *w;
    const float *emb, *out_norm;
    orc_layer *layers;
    float *kc, *vc;     /* [layer][seq][kvh][max_seq][hd] */
    int32_t *len;       /* cached positions per sequence */
    int64_t passes;     /* token positions pushed through the network */
    float *x, *xn, *q, *k, *v, *o, *tmp, *a, *b, *h, *scores;
};

static int cfg_ok(const orc_config *c) {
    if (c->dim <= 0 || c->n_layers <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 ||
        c->head_dim <= 0 || c->hidden <= 0 || c->vocab <= 0 || c->max_seq <= 0 ||
        c->max_batch <= 0)
        return 0;
    if (c->n_heads % c->n_kv_heads) return 0;
    if (c->head_dim % 2) return 0;
    if (c->weight_dtype != ORC_F32 && c->weight_dtype != ORC_BF16 && c->weight_dtype != ORC_Q8) return 0;
    if (c->kv_dtype != ORC_F32 && c->kv_dtype != ORC_BF16) return 0;
    if (!(c->norm_eps >= 0.0f) || !(c->rope_theta > 0.0f)) return 0;
    return 1;
}

size_t orc_weight_count(const orc_config *c) {
    size_t dim = c->dim, qd = (size_t)c->n_heads * c->head_dim,
           kvd = (size_t)c->n_kv_heads * c->head_dim, hid = c->hidden;
    size_t per_layer = dim + qd * dim + 2 * kvd * dim + dim * qd + dim + 3 * hid * dim;
    return (size_t)c->vocab * dim + (size_t)c->n_layers * per_layer + dim;
}

static size_t kv_index(const orc_model *m, int layer, int seq, int kvh, int pos) {
    const orc_config *c = &m->c;
    return ((((size_t)layer * c->max_batch + seq) * c->n_kv_heads + kvh) * c->max_seq + pos) *
           (size_t)c->head_dim;
}

void orc_destroy(orc_model *m) {
    if (!m) return;
    free(m->w);
    free(m->layers);
    free(m->kc);
    free(m->vc);
    free(m->len);
    free(m->x);
    free(m->xn);
    free(m->q);
    free(m->k);
    free(m->v);
    free(m->o);
    free(m->tmp);
    free(m->a);
    free(m->b);
    free(m->h);
    free(m->scores);
    free(m);
}

int orc_create(const orc_config *cfg, const void *weights, size_t nbytes, orc_model **out) {
    if (!cfg || !weights || !out) return ORC_EINVAL;
    *out = NULL;
    if (!cfg_ok(cfg)) return ORC_EINVAL;
    size_t n = orc_weight_count(cfg);
    size_t esz = cfg->weight_dtype == ORC_BF16 ? 2 : 4;
    if (nbytes != n * esz) return ORC_EINVAL;

    orc_model *m = calloc(1, sizeof *m);
    if (!m) return ORC_ENOMEM;
    m->c = *cfg;
    const orc_config *c = &m->c;
    m->w = malloc(n * sizeof(float));
    m->layers = calloc((size_t)c->n_layers, sizeof(orc_layer));
    size_t kvn = (size_t)c->n_layers * c->max_batch * c->n_kv_heads * c->max_seq * c->head_dim;
    m->kc = calloc(kvn, sizeof(float));
    m->vc = calloc(kvn, sizeof(float));
    m->len = calloc((size_t)c->max_batch, sizeof(int32_t));
    size_t qd = (size_t)c->n_heads * c->head_dim, kvd = (size_t)c->n_kv_heads * c->head_dim;
    size_t wide = (size_t)c->dim > qd ? (size_t)c->dim : qd;
    m->x = malloc(wide * sizeof(float));
    m->xn = malloc(wide * sizeof(float));
    m->q = malloc(qd * sizeof(float));
    m->k = malloc(kvd * sizeof(float));
    m->v = malloc(kvd * sizeof(float));
    m->o = malloc(qd * sizeof(float));
    m->tmp = malloc(wide * sizeof(float));
    m->a = malloc((size_t)c->hidden * sizeof(float));
    m->b = malloc((size_t)c->hidden * sizeof(float));
    m->h = malloc((size_t)c->hidden * sizeof(float));
    m->scores = malloc((size_t)c->max_seq * sizeof(float));
    if (!m->w || !m->layers || !m->kc || !m->vc || !m->len || !m->x || !m->xn || !m->q ||
        !m->k || !m->v || !m->o || !m->tmp || !m->a || !m->b || !m->h || !m->scores) {
        orc_destroy(m);
        return ORC_ENOMEM;
    }
    if (cfg->weight_dtype == ORC_BF16) {
        const uint16_t *src = weights;
        for (size_t i = 0; i < n; i++) m->w[i] = orc_bf16_up(src[i]);
    } else {
        memcpy(m->w, weights, n * sizeof(float));
    }
    /* walk the canonical order */
    size_t dim = c->dim, hid = c->hidden;
    const float *p = m->w;
    m->emb = p;
    p += (size_t)c->vocab * dim;
    for (int l = 0; l < c->n_layers; l++) {
        orc_layer *L = &m->layers[l];
        L->attn_norm = p; p += dim;
        L->wq = p; p += qd * dim;
        L->wk = p; p += kvd * dim;
        L->wv = p; p += kvd * dim;
        L->wo = p; p += dim * qd;
        L->ffn_norm = p; p += dim;
        L->w1 = p; p += hid * dim;
        L->w3 = p; p += hid * dim;
        L->w2 = p; p += dim * hid;
    }
    m->out_norm = p;
    if (c->weight_dtype == ORC_Q8) { /* fp32 input weights, quantised matrix by matrix */
        int rc = q8_dequantize_rows((float *)m->emb, (size_t)c->vocab, (int)dim);
        for (int l = 0; l < c->n_layers && rc == ORC_OK; l++) {
            orc_layer *L = &m->layers[l];
            if (rc == ORC_OK) rc = q8_dequantize_rows((float *)L->wq, qd, (int)dim);
            if (rc == ORC_OK) rc = q8_dequantize_rows((float *)L->wk, kvd, (int)dim);
            if (rc == ORC_OK) rc = q8_dequantize_rows((float *)L->wv, kvd, (int)dim);
            if (rc == ORC_OK) rc = q8_dequantize_rows((float *)L->wo, dim, (int)qd);
            if (rc == ORC_OK) rc = q8_dequantize_rows((float *)L->w1, hid, (int)dim);
            if (rc == ORC_OK) rc = q8_dequantize_rows((float *)L->w3, hid, (int)dim);
            if (rc == ORC_OK) rc = q8_dequantize_rows((float *)L->w2, dim, (int)hid);
        }
        if (rc != ORC_OK) {
            orc_destroy(m);
            return rc;
        }
    }
    *out = m;
    return ORC_OK;
}

static float kv_store(const orc_model *m, float x) {
    return m->c.kv_dtype == ORC_BF16 ? orc_bf16_round(x) : x;
}

/* One token at one position through every block; its k and v land in cache slot pos. */
static void forward_token(orc_model *m, int seq, int32_t tok, int pos, float *logits) {
    const orc_config *c = &m->c;
    int dim = c->dim, hd = c->head_dim, H = c->n_heads, KV = c->n_kv_heads;
    int qd = H * hd, kvd = KV * hd, group = H / KV;
    memcpy(m->x, m->emb + (size_t)tok * dim, (size_t)dim * sizeof(float));
    for (int l = 0; l < c->n_layers; l++) {
        const orc_layer *L = &m->layers[l];
        orc_rmsnorm(m->xn, m->x, L->attn_norm, dim, c->norm_eps);
        orc_matvec(m->q, L->wq, m->xn, dim, qd);
        orc_matvec(m->k, L->wk, m->xn, dim, kvd);
        orc_matvec(m->v, L->wv, m->xn, dim, kvd);
        orc_rope(m->q, H, hd, pos, c->rope_theta);
        orc_rope(m->k, KV, hd, pos, c->rope_theta);
        for (int g = 0; g < KV; g++) {
            float *kd = m->kc + kv_index(m, l, seq, g, pos);
            float *vd = m->vc + kv_index(m, l, seq, g, pos);
            for (int i = 0; i < hd; i++) {
                kd[i] = kv_store(m, m->k[g * hd + i]);
                vd[i] = kv_store(m, m->v[g * hd + i]);
            }
        }
        for (int h = 0; h < H; h++) {
            int g = h / group;
            orc_attend(m->o + (size_t)h * hd, m->q + (size_t)h * hd,
                       m->kc + kv_index(m, l, seq, g, 0), m->vc + kv_index(m, l, seq, g, 0),
                       pos + 1, hd, m->scores);
        }
        orc_matvec(m->tmp, L->wo, m->o, qd, dim);
        for (int i = 0; i < dim; i++) m->x[i] = m->x[i] + m->tmp[i];
        orc_rmsnorm(m->xn, m->x, L->ffn_norm, dim, c->norm_eps);
        orc_matvec(m->a, L->w1, m->xn, dim, c->hidden);
        orc_matvec(m->b, L->w3, m->xn, dim, c->hidden);
        orc_silu_mul(m->h, m->a, m->b, c->hidden);
        orc_matvec(m->tmp, L->w2, m->h, c->hidden, dim);
        for (int i = 0; i < dim; i++) m->x[i] = m->x[i] + m->tmp[i];
    }
    if (logits) {
        orc_rmsnorm(m->xn, m->x, m->out_norm, dim, c->norm_eps);
        orc_matvec(logits, m->emb, m->xn, dim, c->vocab);
    }
    m->passes++;
}

int orc_prefill(orc_model *m, int32_t seq, const int32_t *tokens, int32_t n, float *last_logits,
                int32_t *next_id) {
    if (!m || !tokens || n <= 0) return ORC_EINVAL;
    if (seq < 0 || seq >= m->c.max_batch) return ORC_EINVAL;
    if (m->len[seq] != 0) return ORC_ESTATE;
    if (n > m->c.max_seq) return ORC_ECAPACITY;
    for (int i = 0; i < n; i++)
        if (tokens[i] < 0 || tokens[i] >= m->c.vocab) return ORC_EINVAL;
    float *logits = malloc((size_t)m->c.vocab * sizeof(float));
    if (!logits) return ORC_ENOMEM;
    for (int p = 0; p < n; p++) forward_token(m, seq, tokens[p], p, p == n - 1 ? logits : NULL);
    m->len[seq] = n;
    if (last_logits) memcpy(last_logits, logits, (size_t)m->c.vocab * sizeof(float));
    int32_t id = orc_argmax(logits, m->c.vocab);
    free(logits);
    if (next_id) *next_id = id;
    return id < 0 ? ORC_EINVAL : ORC_OK;
}

int orc_decode_step(orc_model *m, int32_t batch, const int32_t *seq_ids, const int32_t *tokens,
                    const int32_t *positions, float *logits, int32_t *next_ids) {
    if (!m || !seq_ids || !tokens || !positions || batch <= 0 || batch > m->c.max_batch)
        return ORC_EINVAL;
    for (int i = 0; i < batch; i++) {
        int s = seq_ids[i];
        if (s < 0 || s >= m->c.max_batch) return ORC_EINVAL;
        for (int j = 0; j < i; j++)
            if (seq_ids[j] == s) return ORC_EINVAL;
        if (tokens[i] < 0 || tokens[i] >= m->c.vocab) return ORC_EINVAL;
        if (positions[i] != m->len[s]) return ORC_EPOS;
        if (positions[i] >= m->c.max_seq) return ORC_ECAPACITY;
    }
    float *row = malloc((size_t)m->c.vocab * sizeof(float));
    if (!row) return ORC_ENOMEM;
    int rc = ORC_OK;
    for (int i = 0; i < batch; i++) {
        int s = seq_ids[i];
        forward_token(m, s, tokens[i], positions[i], row);
        m->len[s] = positions[i] + 1;
        if (logits) memcpy(logits + (size_t)i * m->c.vocab, row, (size_t)m->c.vocab * sizeof(float));
        int32_t id = orc_argmax(row, m->c.vocab);
        if (next_ids) next_ids[i] = id;
        if (id < 0) rc = ORC_EINVAL;
    }
    free(row);
    return rc;
}

int orc_reset(orc_model *m, int32_t seq) {
    if (!m) return ORC_EINVAL;
    if (seq == -1) {
        memset(m->len, 0, (size_t)m->c.max_batch * sizeof(int32_t));
        return ORC_OK;
    }
    if (seq < 0 || seq >= m->c.max_batch) return ORC_EINVAL;
    m->len[seq] = 0;
    return ORC_OK;
}

int32_t orc_seq_len(const orc_model *m, int32_t seq) {
    if (!m || seq < 0 || seq >= m->c.max_batch) return ORC_EINVAL;
    return m->len[seq];
}

int64_t orc_passes(const orc_model *m) { return m ? m->passes : 0; }

int orc_copy_kv(const orc_model *m, int32_t layer, int32_t seq, float *k_out, float *v_out) {
    if (!m || layer < 0 || layer >= m->c.n_layers || seq < 0 || seq >= m->c.max_batch)
        return ORC_EINVAL;
    int n = m->len[seq], hd = m->c.head_dim;
    for (int g = 0; g < m->c.n_kv_heads; g++) {
        size_t dst = (size_t)g * n * hd;
        if (k_out) memcpy(k_out + dst, m->kc + kv_index(m, layer, seq, g, 0), (size_t)n * hd * sizeof(float));
        if (v_out) memcpy(v_out + dst, m->vc + kv_index(m, layer, seq, g, 0), (size_t)n * hd * sizeof(float));
    }
    return n;
}

int orc_layer0_kv(const orc_model *m, int32_t tok, int32_t pos, float *k_out, float *v_out) {
    if (!m || tok < 0 || tok >= m->c.vocab || pos < 0) return ORC_EINVAL;
    const orc_config *c = &m->c;
    int dim = c->dim, kvd = c->n_kv_heads * c->head_dim;
    float *xn = malloc((size_t)dim * sizeof(float));
    if (!xn) return ORC_ENOMEM;
    const orc_layer *L = &m->layers[0];
    orc_rmsnorm(xn, m->emb + (size_t)tok * dim, L->attn_norm, dim, c->norm_eps);
    orc_matvec(k_out, L->wk, xn, dim, kvd);
    orc_matvec(v_out, L->wv, xn, dim, kvd);
    orc_rope(k_out, c->n_kv_heads, c->head_dim, pos, c->rope_theta);
    for (int i = 0; i < kvd; i++) {
        k_out[i] = kv_store(m, k_out[i]);
        v_out[i] = kv_store(m, v_out[i]);
    }
    free(xn);
    return ORC_OK;
}

/*
 * Uncached full recomputation, layer by layer over all n positions at once with a
 * causal mask (position p attends to 0..p).  It keeps its own temporary K/V and
 * leaves the model's cache untouched.  Every output element goes through the same
 * operations in the same order as the cached path, so the two agree bit for bit.
 */
int orc_forward_uncached(orc_model *m, const int32_t *tokens, int32_t n, float *last_logits,
                         int32_t *next_id) {
    if (!m || !tokens || n <= 0) return ORC_EINVAL;
    const orc_config *c = &m->c;
    int dim = c->dim, hd = c->head_dim, H = c->n_heads, KV = c->n_kv_heads, hid = c->hidden;
    int qd = H * hd, kvd = KV * hd, group = H / KV;
    for (int i = 0; i < n; i++)
        if (tokens[i] < 0 || tokens[i] >= c->vocab) return ORC_EINVAL;
    size_t N = (size_t)n;
    float *X = malloc(N * dim * sizeof(float));
    float *XN = malloc(N * dim * sizeof(float));
    float *Q = malloc(N * qd * sizeof(float));
    float *K = malloc(N * kvd * sizeof(float));
    float *V = malloc(N * kvd * sizeof(float));
    float *Kt = malloc(N * kvd * sizeof(float)); /* [kvh][pos][hd] */
    float *Vt = malloc(N * kvd * sizeof(float));
    float *O = malloc(N * qd * sizeof(float));
    float *A = malloc((size_t)hid * sizeof(float));
    float *B = malloc((size_t)hid * sizeof(float));
    float *Hh = malloc((size_t)hid * sizeof(float));
    float *T = malloc((size_t)dim * sizeof(float));
    float *S = malloc(N * sizeof(float));
    float *logits = malloc((size_t)c->vocab * sizeof(float));
    int rc = ORC_OK;
    if (!X || !XN || !Q || !K || !V || !Kt || !Vt || !O || !A || !B || !Hh || !T || !S || !logits) {
        rc = ORC_ENOMEM;
        goto done;
    }
    for (size_t p = 0; p < N; p++)
        memcpy(X + p * dim, m->emb + (size_t)tokens[p] * dim, (size_t)dim * sizeof(float));
    for (int l = 0; l < c->n_layers; l++) {
        const orc_layer *L = &m->layers[l];
        for (size_t p = 0; p < N; p++) {
            orc_rmsnorm(XN + p * dim, X + p * dim, L->attn_norm, dim, c->norm_eps);
            orc_matvec(Q + p * qd, L->wq, XN + p * dim, dim, qd);
            orc_matvec(K + p * kvd, L->wk, XN + p * dim, dim, kvd);
            orc_matvec(V + p * kvd, L->wv, XN + p * dim, dim, kvd);
            orc_rope(Q + p * qd, H, hd, (int)p, c->rope_theta);
            orc_rope(K + p * kvd, KV, hd, (int)p, c->rope_theta);
            for (int g = 0; g < KV; g++)
                for (int i = 0; i < hd; i++) {
                    Kt[((size_t)g * N + p) * hd + i] = kv_store(m, K[p * kvd + (size_t)g * hd + i]);
                    Vt[((size_t)g * N + p) * hd + i] = kv_store(m, V[p * kvd + (size_t)g * hd + i]);
                }
        }
        for (size_t p = 0; p < N; p++)
            for (int h = 0; h < H; h++) {
                int g = h / group;
                orc_attend(O + p * qd + (size_t)h * hd, Q + p * qd + (size_t)h * hd,
                           Kt + (size_t)g * N * hd, Vt + (size_t)g * N * hd, (int)p + 1, hd, S);
            }
        for (size_t p = 0; p < N; p++) {
            float *x = X + p * dim;
            orc_matvec(T, L->wo, O + p * qd, qd, dim);
            for (int i = 0; i < dim; i++) x[i] = x[i] + T[i];
            orc_rmsnorm(XN + p * dim, x, L->ffn_norm, dim, c->norm_eps);
            orc_matvec(A, L->w1, XN + p * dim, dim, hid);
            orc_matvec(B, L->w3, XN + p * dim, dim, hid);
            orc_silu_mul(Hh, A, B, hid);
            orc_matvec(T, L->w2, Hh, hid, dim);
            for (int i = 0; i < dim; i++) x[i] = x[i] + T[i];
        }
    }
    orc_rmsnorm(XN, X + (N - 1) * dim, m->out_norm, dim, c->norm_eps);
    orc_matvec(logits, m->emb, XN, dim, c->vocab);
    m->passes += n;
    if (last_logits) memcpy(last_logits, logits, (size_t)c->vocab * sizeof(float));
    {
        int32_t id = orc_argmax(logits, c->vocab);
        if (next_id) *next_id = id;
        if (id < 0) rc = ORC_EINVAL;
    }
done:
    free(X); free(XN); free(Q); free(K); free(V); free(Kt); free(Vt); free(O);
    free(A); free(B); free(Hh); free(T); free(S); free(logits);
    return rc;
}
