/*
 * ds4_oracle.c -- the plain CPU definition of the ds4 layer step, layer-major
 * prefill, lm_head and sampler.  TEST INFRASTRUCTURE: see ds4_oracle.h for
 * who may use it, the passages it follows and the readings it takes.
 *
 * Every function is the textbook definition written out in double precision,
 * one loop per formula, in the order the pages give the steps.  There is no
 * blocking, fusion or reordering.
 */
#include "ds4_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ formats */

/* IEEE binary16 -> double (exact). */
double orc_f16_value(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int exp = (b >> 10) & 0x1F;
    int man = b & 0x3FF;
    double v;
    if (exp == 0)
        v = ldexp((double)man, -24);                 /* subnormal: man * 2^-24 */
    else if (exp == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(man | 0x400), exp - 25);  /* (1.man) * 2^(exp-15) */
    return sign ? -v : v;
}

/* bfloat16 -> double (exact): the bits are the high half of a binary32. */
double orc_bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* double -> bfloat16, round to nearest, ties to even (8 significant bits). */
uint16_t orc_round_bf16(double x)
{
    if (x == 0.0 || !isfinite(x)) {
        float f = (float)x;
        uint32_t u;
        memcpy(&u, &f, 4);
        return (uint16_t)(u >> 16);
    }
    int e;
    double f = frexp(x, &e);              /* x = f * 2^e, 0.5 <= |f| < 1 */
    double r = nearbyint(ldexp(f, 8));    /* 8 significant bits, ties to even */
    float q = (float)ldexp(r, e - 8);     /* exact in binary32 */
    uint32_t u;
    memcpy(&u, &q, 4);
    return (uint16_t)(u >> 16);
}

static double wval(int dtype, const void *w, size_t i)
{
    if (dtype == ORC_BF16) return orc_bf16_value(((const uint16_t *)w)[i]);
    return (double)((const float *)w)[i];
}

static const void *woff(int dtype, const void *w, size_t elems)
{
    size_t bytes = elems * (dtype == ORC_BF16 ? 2u : 4u);
    return (const char *)w + bytes;
}

/* ------------------------------------------------------------ building blocks */

/* 阶段四 4.1: the token's f16 embedding row, widened. */
void orc_embed(const orc_config *c, const uint16_t *table, int32_t token, double *x)
{
    const uint16_t *row = table + (size_t)token * (size_t)c->hidden;
    for (int i = 0; i < c->hidden; i++) x[i] = orc_f16_value(row[i]);
}

/* RMSNorm: y_i = g_i * x_i / sqrt(mean(x^2) + eps). */
void orc_rmsnorm(int n, const double *x, const float *g, double eps, double *y)
{
    double ss = 0.0;
    for (int i = 0; i < n; i++) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; i++) y[i] = (double)g[i] * x[i] * inv;
}

/* y = W x with W row-major [rows][cols]. */
void orc_matvec(int dtype, const void *w, int rows, int cols, const double *x, double *y)
{
    for (int r = 0; r < rows; r++) {
        double acc = 0.0;
        size_t base = (size_t)r * (size_t)cols;
        for (int j = 0; j < cols; j++) acc += wval(dtype, w, base + j) * x[j];
        y[r] = acc;
    }
}

/* RoPE on one head: pair (2i, 2i+1) rotated by pos * base^(-2i/head_dim). */
void orc_rope(int head_dim, int pos, double base, double *v)
{
    for (int i = 0; i < head_dim / 2; i++) {
        double theta = pow(base, -2.0 * (double)i / (double)head_dim);
        double ang = (double)pos * theta;
        double cs = cos(ang), sn = sin(ang);
        double a = v[2 * i], b = v[2 * i + 1];
        v[2 * i] = a * cs - b * sn;
        v[2 * i + 1] = a * sn + b * cs;
    }
}

/* KV-cache append at position pos, rounded to the storage format. */
void orc_kv_store(const orc_config *c, orc_kv *kv, int pos, const double *k, const double *v)
{
    size_t base = (size_t)pos * (size_t)c->head_dim;
    for (int d = 0; d < c->head_dim; d++) {
        if (c->kv_dtype == ORC_BF16) {
            ((uint16_t *)kv->k)[base + d] = orc_round_bf16(k[d]);
            ((uint16_t *)kv->v)[base + d] = orc_round_bf16(v[d]);
        } else {
            ((float *)kv->k)[base + d] = (float)k[d];
            ((float *)kv->v)[base + d] = (float)v[d];
        }
    }
}

double orc_kv_value(const orc_config *c, const void *cache, int pos, int d)
{
    size_t i = (size_t)pos * (size_t)c->head_dim + (size_t)d;
    if (c->kv_dtype == ORC_BF16) return orc_bf16_value(((const uint16_t *)cache)[i]);
    return (double)((const float *)cache)[i];
}

/* Multi-query attention over the sliding window [max(0, pos-W+1), pos]:
 * every query head uses the one cached K/V head. */
void orc_attention(const orc_config *c, const orc_kv *kv, int pos, const double *q, double *o)
{
    int HD = c->head_dim;
    int lo = pos - c->window + 1;
    if (lo < 0) lo = 0;
    int n = pos - lo + 1;
    double scale = 1.0 / sqrt((double)HD);
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    for (int h = 0; h < c->n_heads; h++) {
        const double *qh = q + (size_t)h * HD;
        double m = -INFINITY;
        for (int j = 0; j < n; j++) {
            double acc = 0.0;
            for (int d = 0; d < HD; d++) acc += qh[d] * orc_kv_value(c, kv->k, lo + j, d);
            s[j] = acc * scale;
            if (s[j] > m) m = s[j];
        }
        double sum = 0.0;
        for (int j = 0; j < n; j++) {
            s[j] = exp(s[j] - m);
            sum += s[j];
        }
        for (int j = 0; j < n; j++) s[j] /= sum;
        for (int d = 0; d < HD; d++) {
            double acc = 0.0;
            for (int j = 0; j < n; j++) acc += s[j] * orc_kv_value(c, kv->v, lo + j, d);
            o[(size_t)h * HD + d] = acc;
        }
    }
    free(s);
}

/* The k largest scores, in descending order; equal scores go to the lower id. */
void orc_topk(const float *s, int n, int k, int32_t *ids)
{
    char *taken = (char *)calloc((size_t)n, 1);
    for (int r = 0; r < k; r++) {
        int best = -1;
        for (int i = 0; i < n; i++) {
            if (taken[i]) continue;
            if (best < 0 || s[i] > s[best]) best = i;
        }
        ids[r] = best;
        taken[best] = 1;
    }
    free(taken);
}

/* Router: scores over all experts, top-k, softmax over the selected scores. */
void orc_router(const orc_config *c, const orc_layer *L, const double *xn2, float *scores,
                int32_t *ids, double *w)
{
    int E = c->n_experts, K = c->top_k;
    double *r = (double *)malloc(sizeof(double) * (size_t)E);
    orc_matvec(c->weight_dtype, L->w_router, E, c->hidden, xn2, r);
    for (int e = 0; e < E; e++) scores[e] = (float)r[e];
    orc_topk(scores, E, K, ids);
    double m = (double)scores[ids[0]], sum = 0.0;
    for (int s = 0; s < K; s++) {
        w[s] = exp((double)scores[ids[s]] - m);
        sum += w[s];
    }
    for (int s = 0; s < K; s++) w[s] /= sum;
    free(r);
}

/* One SwiGLU expert: h = silu(Wg x) * (Wu x); y = Wd h; silu(z) = z / (1 + e^-z). */
void orc_swiglu_expert(const orc_config *c, const void *wg, const void *wu, const void *wd,
                       const double *xn, double *h, double *y)
{
    int H = c->hidden, I = c->expert_inter;
    double *g = (double *)malloc(sizeof(double) * (size_t)I);
    double *u = (double *)malloc(sizeof(double) * (size_t)I);
    orc_matvec(c->weight_dtype, wg, I, H, xn, g);
    orc_matvec(c->weight_dtype, wu, I, H, xn, u);
    for (int i = 0; i < I; i++) h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
    orc_matvec(c->weight_dtype, wd, H, I, h, y);
    free(g);
    free(u);
}

/* 阶段四 4.2: one token through one layer at position pos; x is updated in place
 * and the token's K/V are appended to the layer's cache. */
void orc_layer_step(const orc_config *c, const orc_layer *L, orc_kv *kv, int pos, double *x,
                    orc_trace *t)
{
    orc_layer_step_ids(c, L, kv, pos, x, t, NULL);
}

/* The same layer step with the router's choice given (ids_in: K distinct experts
 * in combine order) instead of the top-k of the scores; their weights are the
 * softmax over their own scores, as orc_router computes them.  NULL: the top-k. */
void orc_layer_step_ids(const orc_config *c, const orc_layer *L, orc_kv *kv, int pos, double *x,
                        orc_trace *t, const int32_t *ids_in)
{
    int H = c->hidden, NH = c->n_heads, HD = c->head_dim, RQ = c->q_rank, RKV = c->kv_rank;
    int E = c->n_experts, K = c->top_k, I = c->expert_inter, dt = c->weight_dtype;
    size_t QD = (size_t)NH * HD;
    double *xn1 = (double *)malloc(sizeof(double) * H);
    double *cq = (double *)malloc(sizeof(double) * RQ);
    double *ckv = (double *)malloc(sizeof(double) * RKV);
    double *q = (double *)malloc(sizeof(double) * QD);
    double *k = (double *)malloc(sizeof(double) * HD);
    double *v = (double *)malloc(sizeof(double) * HD);
    double *o = (double *)malloc(sizeof(double) * QD);
    double *tmp = (double *)malloc(sizeof(double) * H);
    double *xn2 = (double *)malloc(sizeof(double) * H);
    double *moe = (double *)calloc((size_t)H, sizeof(double));
    float *scores = (float *)malloc(sizeof(float) * E);
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * K);
    double *w = (double *)malloc(sizeof(double) * K);
    double *h = (double *)malloc(sizeof(double) * (size_t)(K + 1) * I);

    /* attention half: norm, low-rank Q and KV, RoPE, append, attention, residual */
    orc_rmsnorm(H, x, L->attn_norm, c->rms_eps, xn1);
    orc_matvec(dt, L->wq_a, RQ, H, xn1, cq);
    orc_matvec(dt, L->wq_b, (int)QD, RQ, cq, q);
    orc_matvec(dt, L->wkv_a, RKV, H, xn1, ckv);
    orc_matvec(dt, L->wk_b, HD, RKV, ckv, k);
    orc_matvec(dt, L->wv_b, HD, RKV, ckv, v);
    for (int hh = 0; hh < NH; hh++) orc_rope(HD, pos, c->rope_base, q + (size_t)hh * HD);
    orc_rope(HD, pos, c->rope_base, k);
    orc_kv_store(c, kv, pos, k, v);
    orc_attention(c, kv, pos, q, o);
    orc_matvec(dt, L->wo, H, (int)QD, o, tmp);
    for (int i = 0; i < H; i++) x[i] += tmp[i];
    if (t && t->x_mid) memcpy(t->x_mid, x, sizeof(double) * H);

    /* MoE half: norm, router, top-k, weighted routed experts + shared, residual */
    orc_rmsnorm(H, x, L->ffn_norm, c->rms_eps, xn2);
    orc_router(c, L, xn2, scores, ids, w);
    if (ids_in) {
        double sum = 0.0;
        for (int s = 0; s < K; s++) {
            ids[s] = ids_in[s];
            w[s] = exp((double)scores[ids[s]] - (double)scores[ids[0]]);
            sum += w[s];
        }
        for (int s = 0; s < K; s++) w[s] /= sum;
    }
    for (int s = 0; s < K; s++) {
        size_t e = (size_t)ids[s];
        orc_swiglu_expert(c, woff(dt, L->w_gate, e * I * H), woff(dt, L->w_up, e * I * H),
                          woff(dt, L->w_down, e * H * I), xn2, h + (size_t)s * I, tmp);
        for (int i = 0; i < H; i++) moe[i] += w[s] * tmp[i];
    }
    orc_swiglu_expert(c, L->ws_gate, L->ws_up, L->ws_down, xn2, h + (size_t)K * I, tmp);
    for (int i = 0; i < H; i++) moe[i] += tmp[i];
    for (int i = 0; i < H; i++) x[i] += moe[i];

    if (t) {
        if (t->xn1) memcpy(t->xn1, xn1, sizeof(double) * H);
        if (t->cq) memcpy(t->cq, cq, sizeof(double) * RQ);
        if (t->ckv) memcpy(t->ckv, ckv, sizeof(double) * RKV);
        if (t->q) memcpy(t->q, q, sizeof(double) * QD);
        if (t->k) memcpy(t->k, k, sizeof(double) * HD);
        if (t->v) memcpy(t->v, v, sizeof(double) * HD);
        if (t->attn) memcpy(t->attn, o, sizeof(double) * QD);
        if (t->xn2) memcpy(t->xn2, xn2, sizeof(double) * H);
        if (t->scores) memcpy(t->scores, scores, sizeof(float) * E);
        if (t->ids) memcpy(t->ids, ids, sizeof(int32_t) * K);
        if (t->weights) memcpy(t->weights, w, sizeof(double) * K);
        if (t->h) memcpy(t->h, h, sizeof(double) * (size_t)(K + 1) * I);
        if (t->moe) memcpy(t->moe, moe, sizeof(double) * H);
    }
    free(xn1); free(cq); free(ckv); free(q); free(k); free(v); free(o); free(tmp);
    free(xn2); free(moe); free(scores); free(ids); free(w); free(h);
}

/* 阶段四 4.3: the last layer's output projected to the vocabulary. */
void orc_lm_head(const orc_config *c, const void *lm, const double *x, double *logits)
{
    orc_matvec(c->weight_dtype, lm, c->vocab, c->hidden, x, logits);
}

/* ------------------------------------------------------------------ sampler */

/* Greedy: largest logit, lowest index on ties. */
int32_t orc_argmax(const float *logits, int n)
{
    int best = 0;
    for (int i = 1; i < n; i++)
        if (logits[i] > logits[best]) best = i;
    return best;
}

static const double *g_sort_p;
static int cmp_desc(const void *a, const void *b)
{
    int ia = *(const int *)a, ib = *(const int *)b;
    double pa = g_sort_p[ia], pb = g_sort_p[ib];
    if (pa > pb) return -1;
    if (pa < pb) return 1;
    return (ia > ib) - (ia < ib);
}

/* 阶段四 4.3 sample_full_vocab: temperature, top-p, inverse-CDF walk. */
int32_t orc_sample(const float *logits, int n, double temperature, double top_p, double u,
                   orc_sample_info *info)
{
    return orc_sample_min_p(logits, n, temperature, top_p, 0.0, u, info);
}

int32_t orc_sample_min_p(const float *logits, int n, double temperature, double top_p, double min_p,
                         double u, orc_sample_info *info)
{
    orc_sample_info tmp;
    if (!info) info = &tmp;
    memset(info, 0, sizeof(*info));
    info->minp_margin = 1.0;
    if (temperature <= 0.0) {
        info->n_kept = 1;
        info->cut_sum_margin = info->cut_gap_margin = info->cdf_margin = 1.0;
        return orc_argmax(logits, n);
    }
    double *p = (double *)malloc(sizeof(double) * (size_t)n);
    int *order = (int *)malloc(sizeof(int) * (size_t)n);
    char *kept = (char *)calloc((size_t)n, 1);

    /* 1. temperature scaling, then probabilities relative to the largest */
    double m = -INFINITY;
    for (int i = 0; i < n; i++) {
        p[i] = (double)logits[i] / temperature;
        if (p[i] > m) m = p[i];
    }
    double sum_all = 0.0;
    for (int i = 0; i < n; i++) {
        p[i] = exp(p[i] - m);
        sum_all += p[i];
    }

    /* 2. top-p: descending probability, keep until the cumulative sum reaches top_p */
    for (int i = 0; i < n; i++) order[i] = i;
    g_sort_p = p;
    qsort(order, (size_t)n, sizeof(int), cmp_desc);
    double target = top_p * sum_all;
    int n_kept = n;
    info->cut_index = -1;
    info->cut_next_index = -1;
    if (top_p >= 1.0) {
        for (int i = 0; i < n; i++) kept[i] = 1;
        info->cut_sum_margin = info->cut_gap_margin = 1.0;
    } else {
        double cum = 0.0;
        for (int r = 0; r < n; r++) {
            cum += p[order[r]];
            kept[order[r]] = 1;
            if (cum >= target) {
                n_kept = r + 1;
                double before = cum - p[order[r]];
                double a = fabs(cum - target), b = fabs(target - before);
                info->cut_sum_margin = (a < b ? a : b) / sum_all;
                /* nearest different probability on either side of the crossing
                   token: exact ties are ordered by index everywhere, near-ties
                   are where a lower-precision computation may order differently */
                double pc = p[order[r]], gap = 1.0;
                for (int j = r + 1; j < n; j++)
                    if (p[order[j]] != pc) { gap = (pc - p[order[j]]) / pc; break; }
                for (int j = r - 1; j >= 0; j--)
                    if (p[order[j]] != pc) {
                        double g2 = (p[order[j]] - pc) / pc;
                        if (g2 < gap) gap = g2;
                        break;
                    }
                info->cut_gap_margin = gap;
                info->cut_index = order[r];
                info->cut_next_index = r + 1 < n ? order[r + 1] : -1;
                break;
            }
        }
    }
    /* 3. min-p: of the top-p set, keep the tokens whose probability is at least
       min_p times the largest (p is relative to the largest, which is 1) */
    if (min_p > 0.0)
        for (int i = 0; i < n; i++)
            if (kept[i]) {
                const double mg = fabs(p[i] - min_p) / min_p;
                if (mg < info->minp_margin) info->minp_margin = mg;
                if (p[i] < min_p) kept[i] = 0;
            }
    if (min_p > 0.0) {
        n_kept = 0;
        for (int i = 0; i < n; i++) n_kept += kept[i];
    }
    double sum = 0.0, sq = 0.0;
    for (int i = 0; i < n; i++)
        if (kept[i]) {
            sum += p[i];
            sq += p[i] * p[i];
        }
    info->p_rms = sqrt(sq) / sum;
    info->cut_p = info->cut_index >= 0 ? p[info->cut_index] / sum : 0.0;

    /* 4. inverse CDF in vocabulary order over the kept tokens */
    double rnd = u * sum;
    int32_t id = -1, last = -1;
    for (int i = 0; i < n; i++) {
        if (!kept[i] || p[i] == 0.0) continue;   /* a zero-probability token is never drawn */
        last = i;
        double before = rnd;
        rnd -= p[i];
        if (rnd <= 0.0) {
            id = i;
            info->cdf_margin = (before < -rnd ? before : -rnd) / sum;
            break;
        }
    }
    if (id < 0) {               /* rounding pushed u*sum past the end */
        id = last;
        info->cdf_margin = 0.0;
    }
    info->n_kept = n_kept;
    info->sum_all = sum_all;
    info->sum_kept = sum;
    free(p);
    free(order);
    free(kept);
    return id;
}

/* xorshift64* (Vigna, "An experimental exploration of Marsaglia's xorshift
 * generators, scrambled", 2016): shifts 12, 25, 27 and the published multiplier. */
uint64_t orc_xorshift64s(uint64_t *state)
{
    uint64_t x = *state;
    x ^= x >> 12;
    x ^= x << 25;
    x ^= x >> 27;
    *state = x;
    return x * 0x2545F4914F6CDD1Dull;
}

/* Uniform in [0, 1): the top 24 bits of one draw. */
double orc_uniform(uint64_t *state)
{
    return (double)(orc_xorshift64s(state) >> 40) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------ session */

struct orc_session {
    orc_config c;
    int n_ctx;
    int len;
    int32_t *tokens;
    orc_kv *kv;
};

orc_session *orc_session_new(const orc_config *c, int n_ctx)
{
    if (!c || n_ctx <= 0) return NULL;
    orc_session *s = (orc_session *)calloc(1, sizeof(orc_session));
    s->c = *c;
    s->n_ctx = n_ctx;
    s->tokens = (int32_t *)calloc((size_t)n_ctx, sizeof(int32_t));
    s->kv = (orc_kv *)calloc((size_t)c->n_layers, sizeof(orc_kv));
    size_t esz = c->kv_dtype == ORC_BF16 ? 2u : 4u;
    for (int l = 0; l < c->n_layers; l++) {
        s->kv[l].k = calloc((size_t)n_ctx * c->head_dim, esz);
        s->kv[l].v = calloc((size_t)n_ctx * c->head_dim, esz);
    }
    return s;
}

void orc_session_free(orc_session *s)
{
    if (!s) return;
    for (int l = 0; l < s->c.n_layers; l++) {
        free(s->kv[l].k);
        free(s->kv[l].v);
    }
    free(s->kv);
    free(s->tokens);
    free(s);
}

int orc_session_len(const orc_session *s) { return s->len; }
orc_kv *orc_session_kv(orc_session *s, int layer) { return &s->kv[layer]; }
const int32_t *orc_session_tokens(const orc_session *s) { return s->tokens; }

/* Adopt KV contents the caller wrote through orc_session_kv for positions [0, n). */
int orc_session_restore(orc_session *s, const int32_t *tokens, int n)
{
    if (n < 0 || n >= s->n_ctx) return ORC_ECONTEXT;
    memcpy(s->tokens, tokens, sizeof(int32_t) * (size_t)n);
    s->len = n;
    return ORC_OK;
}

/* 阶段三 prefill_layer_major_cpu: layer l runs over every token of the batch
 * before layer l+1; token t sits at position len + t. */
int orc_prefill(orc_session *s, const orc_model *m, const int32_t *tokens, int n,
                double *logits, double *hidden)
{
    const orc_config *c = &s->c;
    if (n < 0 || (n > 0 && !tokens)) return ORC_EINVAL;
    if (n == 0) return ORC_OK;
    for (int t = 0; t < n; t++)
        if (tokens[t] < 0 || tokens[t] >= c->vocab) return ORC_ETOKEN;
    if (s->len + n >= s->n_ctx) return ORC_ECONTEXT;   /* 阶段一: tokens >= context */
    int H = c->hidden;
    double *X = (double *)malloc(sizeof(double) * (size_t)n * H);
    for (int t = 0; t < n; t++) orc_embed(c, m->tok_embd, tokens[t], X + (size_t)t * H);
    for (int l = 0; l < c->n_layers; l++)
        for (int t = 0; t < n; t++)
            orc_layer_step(c, &m->layers[l], &s->kv[l], s->len + t, X + (size_t)t * H, NULL);
    memcpy(s->tokens + s->len, tokens, sizeof(int32_t) * (size_t)n);
    s->len += n;
    if (logits) orc_lm_head(c, m->lm_head, X + (size_t)(n - 1) * H, logits);
    if (hidden) memcpy(hidden, X, sizeof(double) * (size_t)n * H);
    free(X);
    return ORC_OK;
}

/* 阶段四: one generated token through every layer. */
int orc_decode_step(orc_session *s, const orc_model *m, int32_t token, double *logits,
                    double *hidden)
{
    return orc_prefill(s, m, &token, 1, logits, hidden);
}

/* ds4_session_common_prefix: leading tokens shared by the live history and a prompt. */
int orc_common_prefix(const orc_session *s, const int32_t *tokens, int n)
{
    int i = 0;
    while (i < n && i < s->len && s->tokens[i] == tokens[i]) i++;
    return i;
}

/* Keep the KV of the first common_prefix positions; later ones are dead. */
int orc_truncate(orc_session *s, int common_prefix)
{
    if (common_prefix < 0 || common_prefix > s->len) return ORC_EINVAL;
    s->len = common_prefix;
    return ORC_OK;
}
