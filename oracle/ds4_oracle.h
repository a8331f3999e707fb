/*
 * ds4_oracle.h -- plain, slow, single-threaded CPU definition of the ds4 layer
 * step, layer-major prefill, lm_head and sampler.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code with
 * the CUDA library.
 *
 * What it follows (page "ds4.c 学习笔记 -- 端到端推理流程"):
 *   - 阶段四 4.1 (embed_token_f16): an f16 embedding row widened to float.
 *   - 阶段四 4.2 (单层前向 pseudocode): RMSNorm -> low-rank Q/KV projection ->
 *     RoPE -> KV-cache append -> 64-head MQA over a 128-token window ->
 *     residual -> RMSNorm -> router over 256 experts -> top-6 -> weighted
 *     experts + shared expert -> residual.
 *   - 阶段四 4.3 (sample_full_vocab snippet): lm_head to logits, temperature
 *     scaling, top-p filter by descending probability, inverse-CDF walk
 *     `rnd = u * sum; rnd -= p_i; if (rnd <= 0) return i`, argmax as T -> 0.
 *   - 阶段三 (prefill_layer_major_cpu figure): every layer over the whole token
 *     batch before the next layer; after prefill every context K/V is cached.
 *   - 阶段一 (request_exceeds_context): prompts with tokens >= context rejected.
 * and page "【#5】ds4.c を読み解く" section 3 (ds4_session_common_prefix /
 * ds4_session_sync): keep the KV of the common prefix, prefill only the suffix.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   RMSNorm eps = 1e-6; RoPE on adjacent pairs (2i, 2i+1) of the whole head,
 *   theta_i = base^(-2i/head_dim); K cached after RoPE; the window holds the
 *   current token and the W-1 before it; score scale 1/sqrt(head_dim); an
 *   output projection W_o (64*128 != 4096); router top-k on raw scores, ties to
 *   the lower expert id, weights = softmax over the selected scores; shared
 *   expert added with weight 1; no final norm before lm_head; sampler ties
 *   in the top-p order go to the lower token id, the crossing token is kept,
 *   dropped and zero-probability tokens are skipped by the walk.
 *
 * Arithmetic is double precision throughout.  Values that the method stores
 * in a narrower format are rounded to it where they are stored: the KV cache
 * (bf16 or f32, by configuration); router scores and logits are rounded to
 * float before the integer decisions taken on them (top-k, argmax), which is
 * the precision the decisions are taken in.
 */
#ifndef DS4_ORACLE_H
#define DS4_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_OK = 0, ORC_EINVAL = -1, ORC_ECONTEXT = -2, ORC_ETOKEN = -3 };

typedef struct {
    int n_layers, hidden, n_heads, head_dim, q_rank, kv_rank, window;
    int n_experts, top_k, expert_inter, vocab;
    double rope_base, rms_eps;
    int weight_dtype;   /* ORC_F32 or ORC_BF16: all matrices incl. lm_head */
    int kv_dtype;       /* ORC_F32 or ORC_BF16: KV-cache storage */
} orc_config;

/* One layer's weights, row-major [out][in].  bf16 matrices are uint16 bits. */
typedef struct {
    const float *attn_norm;   /* [H] */
    const void *wq_a;         /* [RQ][H] */
    const void *wq_b;         /* [NH*HD][RQ] */
    const void *wkv_a;        /* [RKV][H] */
    const void *wk_b;         /* [HD][RKV] */
    const void *wv_b;         /* [HD][RKV] */
    const void *wo;           /* [H][NH*HD] */
    const float *ffn_norm;    /* [H] */
    const void *w_router;     /* [E][H] */
    const void *w_gate;       /* [E][I][H] */
    const void *w_up;         /* [E][I][H] */
    const void *w_down;       /* [E][H][I] */
    const void *ws_gate;      /* [I][H] */
    const void *ws_up;        /* [I][H] */
    const void *ws_down;      /* [H][I] */
} orc_layer;

typedef struct {
    const uint16_t *tok_embd; /* f16 bits [V][H] */
    const void *lm_head;      /* [V][H] */
    const orc_layer *layers;  /* [n_layers] */
} orc_model;

/* One layer's KV cache in its storage format: [n_ctx][HD] each. */
typedef struct {
    void *k;
    void *v;
} orc_kv;

/* Optional intermediate values of one layer step; any pointer may be NULL. */
typedef struct {
    double *xn1;      /* [H]      normalised input */
    double *cq;       /* [RQ]     Q latent */
    double *ckv;      /* [RKV]    KV latent */
    double *q;        /* [NH*HD]  queries after RoPE */
    double *k;        /* [HD]     key after RoPE (before storage rounding) */
    double *v;        /* [HD]     value (before storage rounding) */
    double *attn;     /* [NH*HD]  attention output, head-major */
    double *x_mid;    /* [H]      residual after attention */
    double *xn2;      /* [H]      normalised residual for the MoE */
    float *scores;    /* [E]      router scores */
    int32_t *ids;     /* [K]      selected experts, descending score */
    double *weights;  /* [K]      softmax over the selected scores */
    double *h;        /* [(K+1)*I] SwiGLU hidden, routed slots then shared */
    double *moe;      /* [H]      expert output added to the residual */
} orc_trace;

typedef struct {
    int n_kept;             /* tokens kept by the top-p filter */
    double sum_all;         /* sum of p over the vocabulary (p relative to the max) */
    double sum_kept;        /* sum of p over kept tokens */
    double cut_sum_margin;  /* distance of the top-p target from the cumulative sums
                               on both sides of the crossing token, / sum_all */
    double cut_gap_margin;  /* relative p gap between the crossing token and the nearest
                               token of different probability on either side */
    double cdf_margin;      /* distance of u*sum_kept from the selected token's CDF
                               interval ends, / sum_kept */
    int cut_index;          /* vocabulary id of the crossing token (-1: all kept) */
    int cut_next_index;     /* vocabulary id of the token after it in top-p order */
    double cut_p;           /* its probability, / sum_kept */
    double p_rms;           /* sqrt(sum of kept p^2) / sum_kept: scale of how far a
                               cumulative sum moves when every p carries a small
                               independent relative error */
    double minp_margin;     /* min-p: smallest |p - min_p| / min_p over the top-p set
                               (1 when min-p is off) */
} orc_sample_info;

/* ---- scalar formats ---- */
double orc_f16_value(uint16_t bits);
double orc_bf16_value(uint16_t bits);
uint16_t orc_round_bf16(double x);

/* ---- building blocks ---- */
void orc_embed(const orc_config *c, const uint16_t *table, int32_t token, double *x);
void orc_rmsnorm(int n, const double *x, const float *g, double eps, double *y);
void orc_matvec(int dtype, const void *w, int rows, int cols, const double *x, double *y);
void orc_rope(int head_dim, int pos, double base, double *v);
void orc_kv_store(const orc_config *c, orc_kv *kv, int pos, const double *k, const double *v);
double orc_kv_value(const orc_config *c, const void *cache, int pos, int d);
void orc_attention(const orc_config *c, const orc_kv *kv, int pos, const double *q, double *o);
void orc_topk(const float *s, int n, int k, int32_t *ids);
void orc_router(const orc_config *c, const orc_layer *L, const double *xn2, float *scores,
                int32_t *ids, double *w);
void orc_swiglu_expert(const orc_config *c, const void *wg, const void *wu, const void *wd,
                       const double *xn, double *h, double *y);
void orc_layer_step(const orc_config *c, const orc_layer *L, orc_kv *kv, int pos, double *x,
                    orc_trace *t);
/* orc_layer_step with the router's choice given: ids (K distinct experts, combine
 * order) replace the top-k; the weights are the softmax over their scores.  For
 * checking a result whose k-th and (k+1)-th scores lie within rounding of each
 * other, where either choice is the method's result.  ids == NULL: orc_layer_step. */
void orc_layer_step_ids(const orc_config *c, const orc_layer *L, orc_kv *kv, int pos, double *x,
                        orc_trace *t, const int32_t *ids);
void orc_lm_head(const orc_config *c, const void *lm, const double *x, double *logits);

/* ---- sampler ---- */
int32_t orc_argmax(const float *logits, int n);
int32_t orc_sample(const float *logits, int n, double temperature, double top_p, double u,
                   orc_sample_info *info);
/* The same with a min-p filter (reading of the pages' sample_top_p_min_p, which
 * names the two filters only): a token of the top-p set is kept if its probability
 * is at least min_p times the largest; min_p <= 0 is off. */
int32_t orc_sample_min_p(const float *logits, int n, double temperature, double top_p, double min_p,
                         double u, orc_sample_info *info);
uint64_t orc_xorshift64s(uint64_t *state);
double orc_uniform(uint64_t *state);

/* ---- session: KV cache, token history, prefill, decode, truncate ---- */
typedef struct orc_session orc_session;
orc_session *orc_session_new(const orc_config *c, int n_ctx);
void orc_session_free(orc_session *s);
int orc_session_len(const orc_session *s);
orc_kv *orc_session_kv(orc_session *s, int layer);
const int32_t *orc_session_tokens(const orc_session *s);
int orc_session_restore(orc_session *s, const int32_t *tokens, int n);
int orc_prefill(orc_session *s, const orc_model *m, const int32_t *tokens, int n,
                double *logits /* [V] of the last token, may be NULL */,
                double *hidden /* [n][H] final hidden states, may be NULL */);
int orc_decode_step(orc_session *s, const orc_model *m, int32_t token, double *logits,
                    double *hidden /* [H], may be NULL */);
int orc_common_prefix(const orc_session *s, const int32_t *tokens, int n);
int orc_truncate(orc_session *s, int common_prefix);

#ifdef __cplusplus
}
#endif
#endif
