/*
 * ds4g.h -- C ABI of the GB300 (sm_103a) implementation of the ds4 per-token
 * layer step, its layer-major batched form for prefill, the lm_head and the
 * temperature / top-p sampler.
 *
 * Sources of the operations (cited by page title and section):
 *   [P3] "ds4.c 学习笔记 -- 端到端推理流程" (ds4-learning.pages.dev/inference-pipeline)
 *        阶段一  request_exceeds_context: a prompt with tokens >= context is rejected.
 *        阶段三  ds4_session_sync -> prefill_layer_major_cpu: reuse the cached prefix,
 *                then run every layer over the whole token batch before the next.
 *        阶段四  4.1 embed_token_f16; 4.2 the single-layer forward pseudocode
 *                (RMSNorm, low-rank Q/KV, RoPE, KV append, 64-head MQA over a
 *                128-token window, residual, RMSNorm, router over 256 experts,
 *                top-6, weighted experts plus a shared expert, residual),
 *                run once per layer per decoded token; 4.3 lm_head to 129280
 *                logits and sample_full_vocab (temperature, top-p, inverse CDF).
 *   [P1] "【#5】ds4.c を読み解く" (qiita.com/yoshiyakato) section 2: one worker owns
 *        the session and its KV; section 3: ds4_session_common_prefix and
 *        ds4_session_sync keep the KV of the common prefix and prefill the suffix.
 *
 * Conventions.
 *  - Every call returns an int status: DS4G_OK (0) or a negative DS4G_E* code;
 *    ds4g_sample returns the token id (>= 0) or a negative code.
 *  - Memory: the library never allocates device memory.  Weights are caller-owned
 *    device buffers that must outlive the model; a session lives inside one
 *    caller-owned device buffer of ds4g_session_bytes() bytes (KV cache, RoPE
 *    table, activations, logits).  Host-side bookkeeping (token history) is
 *    allocated with malloc and freed by the destroy calls.
 *  - Streams: every device operation of a session is issued on the stream
 *    given at ds4g_session_create, in call order.  Calls that return data to the
 *    host (ds4g_sample, ds4g_session_router) synchronise that stream.  A session
 *    of a model with the tensor-core prefill also owns one stream and two events
 *    of its own (created with the session, destroyed with it): each layer's shared
 *    expert GEMMs run on that stream, forked from and joined back into the
 *    session stream within the same ds4g_prefill call, so the ordering the caller
 *    sees is unchanged.
 *  - Threads: a session has one owner thread ([P1] section 2); the library is not
 *    thread-safe per session.  Different sessions may run on different threads.
 *  - Layouts are row-major [out][in] ("W x" is a dot product of each row with x).
 *    bf16 tensors hold raw bfloat16 bits; the embedding table is IEEE binary16.
 *  - Errors leave the session unchanged unless stated otherwise; DS4G_ECUDA
 *    reports a failed launch or CUDA call, after which the session is undefined.
 */
#ifndef DS4G_H
#define DS4G_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { DS4G_F32 = 0, DS4G_BF16 = 1 };

enum {
    DS4G_OK = 0,
    DS4G_EINVAL = -1,    /* bad argument, shape or handle */
    DS4G_ECONTEXT = -2,  /* the tokens would not fit: len + n >= n_ctx ([P3] 阶段一) */
    DS4G_ETOKEN = -3,    /* a token id outside [0, vocab) */
    DS4G_ECUDA = -4,     /* a CUDA call or kernel launch failed */
    DS4G_ETIMEOUT = -5,  /* a bounded device-side wait gave up */
    DS4G_ESIZE = -6,     /* a caller buffer is too small */
    DS4G_ENONFINITE = -7 /* a router score was NaN or infinite (the hidden state is not
                            finite); the step's results are invalid */
};

/* Model shape and formats.  The five synthetic workloads use hidden 4096,
 * 64 heads x 128, q_rank 1024, kv_rank 512, window 128, 256 experts top-6,
 * expert_inter 1024, vocab 129280 (and a tiny FP32 variant). */
typedef struct {
    int n_layers;
    int hidden;        /* H */
    int n_heads;       /* NH query heads; one shared K/V head (MQA) */
    int head_dim;      /* HD, even */
    int q_rank;        /* RQ: Q low-rank latent */
    int kv_rank;       /* RKV: KV low-rank latent */
    int window;        /* W: attention covers positions [pos-W+1, pos] */
    int n_experts;     /* E routed experts */
    int top_k;         /* K experts per token (<= 8) */
    int expert_inter;  /* I: SwiGLU inner width of every expert, shared one included */
    int vocab;         /* V */
    float rope_base;   /* RoPE base; pair (2i, 2i+1) turns by pos * base^(-2i/HD) */
    float rms_eps;     /* RMSNorm epsilon inside the square root */
    int weight_dtype;  /* DS4G_BF16 or DS4G_F32, all matrices including lm_head */
    int kv_dtype;      /* DS4G_BF16 or DS4G_F32, KV-cache storage */
    int prefill_chunk; /* tokens per layer-major pass (0: 4096); sets workspace size */
    int decode_kernel; /* DS4G_DECODE_AUTO: one persistent launch per decode step when
                          the device supports cooperative launch, else one kernel per
                          stage; DS4G_DECODE_STAGED forces one kernel per stage */
    int prefill_kernel; /* DS4G_PREFILL_AUTO: tensor-core GEMMs (tcgen05, BF16
                           activations times BF16 weights, FP32 accumulation and FP32
                           residual; the router's input as a BF16 hi/lo pair, so that its
                           scores carry about 16 significant bits of the normalised
                           residual) when the weights are BF16 and every weight piece is a
                           multiple of 128 rows (64 for expert gate/up) and every
                           reduction a multiple of 64, else SIMT GEMMs with FP32
                           activations; DS4G_PREFILL_HILO: the same tensor-core GEMMs
                           with every activation as a BF16 hi/lo pair (twice the tensor
                           work); DS4G_PREFILL_SIMT forces the SIMT GEMMs */
} ds4g_config;

enum { DS4G_DECODE_AUTO = 0, DS4G_DECODE_STAGED = 1 };
enum { DS4G_PREFILL_AUTO = 0, DS4G_PREFILL_SIMT = 1, DS4G_PREFILL_HILO = 2 };

/* One layer's weights (device pointers).  Gains are f32; matrices weight_dtype. */
typedef struct {
    const void *attn_norm; /* [H]          RMSNorm gain before attention */
    const void *wq_a;      /* [RQ][H]      Q down-projection */
    const void *wq_b;      /* [NH*HD][RQ]  Q up-projection, head-major rows */
    const void *wkv_a;     /* [RKV][H]     KV down-projection */
    const void *wk_b;      /* [HD][RKV]    K up-projection */
    const void *wv_b;      /* [HD][RKV]    V up-projection */
    const void *wo;        /* [H][NH*HD]   attention output projection */
    const void *ffn_norm;  /* [H]          RMSNorm gain before the MoE */
    const void *w_router;  /* [E][H]       router scores */
    const void *w_gate;    /* [E][I][H]    routed experts' gate projections */
    const void *w_up;      /* [E][I][H]    routed experts' up projections */
    const void *w_down;    /* [E][H][I]    routed experts' down projections */
    const void *ws_gate;   /* [I][H]       shared expert */
    const void *ws_up;     /* [I][H] */
    const void *ws_down;   /* [H][I] */
} ds4g_layer_weights;

typedef struct {
    const void *tok_embd;               /* f16 [V][H] */
    const void *lm_head;                /* [V][H] */
    const ds4g_layer_weights *layers;   /* host array of n_layers entries (copied) */
} ds4g_weights;

typedef struct ds4g_model ds4g_model;
typedef struct ds4g_session ds4g_session;

/* Validate the shape and record the weight pointers (copied; no device work
 * beyond setting kernel attributes).  DS4G_EINVAL if a dimension is unsupported:
 * H, RQ, RKV, I and HD must be multiples of 8, HD <= 256, W in [1, 1024],
 * top_k in [1, 8] and <= n_experts, n_experts <= 1024 and a multiple of 4, the
 * K/V window (2 W HD elements) and each activation vector must fit in 227 KB of
 * shared memory; or if a pointer is NULL or not 16-byte aligned. */
int ds4g_model_create(const ds4g_config *cfg, const ds4g_weights *w, ds4g_model **out);
void ds4g_model_destroy(ds4g_model *m);

/* Device bytes a session of context n_ctx needs (0 on a bad argument). */
size_t ds4g_session_bytes(const ds4g_config *cfg, int n_ctx);

/* Lay a session out in dev_mem (256-byte aligned, >= ds4g_session_bytes) and
 * fill its RoPE table on `cuda_stream` (a cudaStream_t; NULL = legacy stream).
 * The session starts empty (len 0).  DS4G_ESIZE if bytes is too small; DS4G_ECUDA
 * if its side stream or events cannot be created (tensor-core prefill). */
int ds4g_session_create(ds4g_model *m, int n_ctx, void *dev_mem, size_t bytes,
                        void *cuda_stream, ds4g_session **out);
void ds4g_session_destroy(ds4g_session *s);

/* [P3] 阶段三 / 阶段四: append n tokens (host array) at positions [len, len+n)
 * with layer-major prefill; afterwards every K/V of the context is cached and
 * the logits of the last token are at ds4g_session_logits.  n == 0 is a no-op.
 * DS4G_ECONTEXT if len + n >= n_ctx, DS4G_ETOKEN if a token is out of range. */
int ds4g_prefill(ds4g_session *s, const int32_t *tokens, int n);

/* [P3] 阶段四: one token through every layer (4.2, once per layer), then the
 * lm_head (4.3).  Same errors as ds4g_prefill with n = 1. */
int ds4g_decode_step(ds4g_session *s, int32_t token);

/* [P3] 阶段四 4.2 without 4.3: one token through every layer, no lm_head (for
 * callers that need the KV cache and the final hidden state but not the logits).
 * The final hidden state is at ds4g_session_hidden; the logits are not updated.
 * Same errors as ds4g_decode_step. */
int ds4g_decode_layers(ds4g_session *s, int32_t token);

/* ds4g_decode_layers with the final hidden state returned to the caller:
 * hidden_host (host memory, hidden floats) holds it when the call returns.  Pinned
 * (page-locked) memory is written by the persistent decode kernel itself through its
 * device view, and the kernel's last CTA signals completion through a pinned word of
 * the session (64 bytes of pinned host memory, allocated on first use and freed by
 * ds4g_session_destroy); the call returns on that signal, while the kernel may still
 * be exiting (later work on the session stream is ordered after it).  Other memory
 * gets a device-to-host copy and a stream synchronisation.  DS4G_ETIMEOUT if the
 * kernel gave up a wait (see ds4g_session_status).  One call per token for a host
 * loop that consumes the hidden state.  DS4G_EINVAL if
 * hidden_host is NULL; otherwise the errors of ds4g_decode_step (the session is
 * unchanged on DS4G_ETOKEN / DS4G_ECONTEXT). */
int ds4g_decode_layers_host(ds4g_session *s, int32_t token, float *hidden_host);

/* [P3] 阶段四 4.2 + 4.3 in one call: token through every layer and the lm_head
 * (as ds4g_decode_step), then the next token drawn from the logits (as
 * ds4g_sample, with its workspace, temperature, top_p and rng_state rules).
 * Returns the drawn token id (>= 0) or a negative DS4G_* code; the call
 * synchronises the session stream.  The one call per generated token of a
 * sampling loop. */
int32_t ds4g_decode_sample(ds4g_session *s, int32_t token, float temperature, float top_p,
                           uint64_t *rng_state, void *workspace, size_t workspace_bytes);

/* [P1] section 3 ds4_session_common_prefix: number of leading tokens shared by
 * the session's history and tokens[0..n). */
int ds4g_session_common_prefix(const ds4g_session *s, const int32_t *tokens, int n);

/* [P1] section 3 / [P3] 阶段三: keep the cached K/V of positions
 * [0, common_prefix); later positions become dead and are overwritten by the
 * next prefill.  0 <= common_prefix <= len, else DS4G_EINVAL; equal to len is a
 * no-op.  The logits are not recomputed. */
int ds4g_session_truncate(ds4g_session *s, int common_prefix);

/* [P1] section 3 ds4_session_sync / [P3] 阶段三: bring the session to the prompt
 * tokens[0..n) (host) in one call.  The cached K/V of the prompt's common prefix
 * with the history is kept, the rest is dropped, and the suffix is prefilled,
 * so that the session then holds exactly the prompt and the logits of its last
 * token.  The logits of a token are not kept once later tokens were processed,
 * so a prompt that the history already holds (whole, or as a prefix) runs its
 * last token again.  n == 0 empties the session.  *n_prefilled (may be NULL)
 * receives the number of tokens run through the layers.  Checked before the
 * session changes: DS4G_ECONTEXT if n >= n_ctx, DS4G_ETOKEN if a token is out of
 * range; then the errors of ds4g_prefill. */
int ds4g_session_sync(ds4g_session *s, const int32_t *tokens, int n, int *n_prefilled);

/* [P1] section 6 ds4_session_rewrite_from_common: rewrite the live checkpoint to
 * the prompt tokens[0..n) from a common prefix the caller found with
 * ds4g_session_common_prefix: positions [0, common) are kept and tokens[common..n)
 * are prefilled (when n > common; else the session is cut to n).  A prompt equal
 * to the history (common == n == len) changes nothing.  DS4G_EINVAL unless
 * 0 <= common <= ds4g_session_common_prefix(s, tokens, n); ECONTEXT and ETOKEN as
 * for ds4g_session_sync, checked before the session changes. */
int ds4g_session_rewrite_from_common(ds4g_session *s, const int32_t *tokens, int n, int common);

int ds4g_session_len(const ds4g_session *s);

/* Device pointer to the f32 [V] logits of the last processed token. */
const float *ds4g_session_logits(const ds4g_session *s);

/* Device pointer to the f32 [H] final hidden state (last layer's output) of the
 * last processed token. */
const float *ds4g_session_hidden(const ds4g_session *s);

/* Device pointers of layer `layer`'s K and V caches: [n_ctx][HD] of kv_dtype,
 * K stored after RoPE.  For tests and for restoring a saved cache. */
int ds4g_session_kv(ds4g_session *s, int layer, void **k, void **v);

/* Adopt K/V contents the caller wrote for positions [0, n) with the token
 * history tokens[0..n) (host): a restore of a saved cache.  DS4G_ECONTEXT if
 * n >= n_ctx. */
int ds4g_session_restore(ds4g_session *s, const int32_t *tokens, int n);

/* [P1] section 3 (steps 3-4: the disk KV cache, whose payload is restored before
 * only the suffix is prefilled): a checkpoint of a session's cached state, the
 * token history and the K/V rows of positions [0, len) of every layer, in a
 * caller-owned host buffer.  Layout (little-endian): a 64-byte header (magic
 * "DS4GKV01", format version, K/V element size, n_layers, head_dim, token count,
 * a digest of the configuration), the int32 tokens padded to 16 bytes, then per
 * layer the K rows and the V rows, [len][head_dim] each, as cached (K after RoPE).
 * The logits are not part of it: after a load, ds4g_session_sync with the prompt
 * runs the suffix (at least the last token) again. */
size_t ds4g_checkpoint_bytes(const ds4g_config *cfg, int n_tokens);
/* Write the checkpoint of s into buf (host memory of `bytes` bytes; pinned
 * memory copies faster).  Synchronises the session stream.  DS4G_ESIZE if bytes <
 * ds4g_checkpoint_bytes(cfg, len). */
int ds4g_session_save(ds4g_session *s, void *buf, size_t bytes);
/* Replace the state of s by a checkpoint written by ds4g_session_save for a model
 * of the same configuration: DS4G_EINVAL on a header or configuration mismatch,
 * DS4G_ESIZE if bytes is shorter than the checkpoint, DS4G_ECONTEXT if its length
 * is >= n_ctx, DS4G_ETOKEN if a token is out of range; the session is unchanged on
 * any of these.  If a copy to the device fails (DS4G_ECUDA), some layers' K/V rows
 * may already be overwritten, so the session is emptied (len 0).  Synchronises the
 * session stream. */
int ds4g_session_load(ds4g_session *s, const void *buf, size_t bytes);

/* Router decision of the last decoded token: ids (int32) and weights (f32) of
 * `layer`, top_k each, copied to host arrays (synchronises the stream). */
int ds4g_session_router(ds4g_session *s, int layer, int32_t *ids, float *weights);

/* Device pointer of one decode-step intermediate (the last layer's values of
 * the last ds4g_decode_step), for element-wise checks; NULL if unknown. */
enum {
    DS4G_DBG_X = 0,       /* f32 [H] residual after the step (layer output) */
    DS4G_DBG_CQKV = 1,    /* f32 [RQ+RKV] Q and KV latents */
    DS4G_DBG_Q = 2,       /* f32 [NH*HD] queries after RoPE */
    DS4G_DBG_ATTN = 3,    /* f32 [NH*HD] attention output, head-major */
    DS4G_DBG_XMID = 4,    /* f32 [H] residual after the attention half */
    DS4G_DBG_XN2 = 5,     /* f32 [H] normalised residual entering the MoE */
    DS4G_DBG_SCORES = 6,  /* f32 [E] router scores */
    DS4G_DBG_H = 7,       /* f32 [(K+1)*I] SwiGLU hidden, routed slots then shared */
    DS4G_DBG_HIDDEN = 8,  /* f32 [H] final hidden state (same as DS4G_DBG_X) */
    DS4G_DBG_PREFILL_X = 9, /* f32 [prefill_chunk][H] final hidden states of the last
                               prefill chunk (row t = t-th token of that chunk) */
    DS4G_DBG_STATUS = 10,   /* int32 raw device status word (0: no device-side error) */
    DS4G_DBG_PREFILL_LAYER_X = 11 /* f32 [L+1][H]: the last prefilled token's residual
                                     entering each layer, then its final hidden state */
};
const void *ds4g_session_debug(const ds4g_session *s, int which);

/* Record the residual stream at chosen positions, for teacher-forced checks of a
 * layer against a reference ([P3] 阶段四 4.2: each layer maps the residual x of a
 * position to the next layer's x).  positions: host array of n absolute session
 * positions (copied; 0 <= position < n_ctx; n <= 64).  buf: device memory owned by
 * the caller, n * (n_layers + 1) * hidden floats, which must outlive the setting.
 * Whenever a later ds4g_prefill, ds4g_decode_step or ds4g_decode_layers computes
 * positions[i], row i * (n_layers + 1) + l of buf receives the residual entering
 * layer l (row l = 0: the widened embedding), and row l = n_layers the final
 * hidden state.  n = 0 turns recording off.  DS4G_EINVAL on a bad argument; the
 * setting is then unchanged.  Recording adds device-to-device copies to a prefill
 * and one store per element to a decode step. */
int ds4g_session_set_probe(ds4g_session *s, const int32_t *positions, int n, float *buf);

/* Synchronise the session stream and report the first device-side error since the
 * last call: DS4G_ETIMEOUT (a bounded wait gave up) or DS4G_ENONFINITE (a router
 * score was not finite; the expert choice then falls back to the lowest unused
 * ids, so every access stays in bounds).  The step's results are then invalid.
 * The flag is cleared.  DS4G_ECUDA if the stream reports an error. */
int ds4g_session_status(ds4g_session *s);

/* Kernels this session has launched so far (all calls on it). */
uint64_t ds4g_session_launches(const ds4g_session *s);

/* Tracing: per-kernel timing.  While on, decode steps run one kernel per stage,
 * every kernel is bracketed by CUDA events on the session stream and the step
 * synchronises the stream at its end; a tensor-core prefill records an event after
 * every launch of each chunk, synchronises at the chunk's end and charges each
 * launch the time since the previous event (timing removes the overlap that
 * programmatic dependent launch gives consecutive kernels).  ds4g_session_timing
 * copies the accumulated milliseconds and launch counts of each kernel kind
 * (DS4G_K_*) into ms[0..n) and counts[0..n), then resets them. */
enum {
    DS4G_K_QKV_A = 0,      /* RMSNorm + Q/KV down-projections */
    DS4G_K_QKV_B = 1,      /* Q/K/V up-projections + RoPE + KV append */
    DS4G_K_ATTN = 2,       /* sliding-window MQA */
    DS4G_K_WO = 3,         /* output projection + residual */
    DS4G_K_ROUTER = 4,     /* RMSNorm + router + top-k */
    DS4G_K_EXPERT_GU = 5,  /* routed + shared gate/up with SwiGLU */
    DS4G_K_EXPERT_DOWN = 6,/* down projections + combine + residual */
    DS4G_K_LM_HEAD = 7,
    /* tensor-core prefill ([P3] 阶段三, layer-major) */
    DS4G_K_P_EMBED = 8,       /* embedding rows */
    DS4G_K_P_NORM = 9,        /* RMSNorm rows (the first layer's attention norm, every FFN norm) */
    DS4G_K_P_QKV_A = 10,      /* [W_qa; W_kva] GEMM */
    DS4G_K_P_Q_B = 11,        /* W_qb GEMM + RoPE */
    DS4G_K_P_KV_B = 12,       /* [W_kb; W_vb] GEMM + RoPE + K/V append */
    DS4G_K_P_ATTN = 13,       /* windowed attention */
    DS4G_K_P_WO = 14,         /* W_o GEMM + residual */
    DS4G_K_P_ROUTER = 15,     /* router GEMM */
    DS4G_K_P_TOPK = 16,       /* top-k + softmax of the selected scores */
    DS4G_K_P_GROUP = 17,      /* grouping of (token, slot) entries by expert */
    DS4G_K_P_GATE_UP = 18,    /* routed gate/up GEMM + SwiGLU */
    DS4G_K_P_SHARED_GU = 19,  /* shared expert gate/up GEMM + SwiGLU */
    DS4G_K_P_DOWN = 20,       /* routed down GEMM */
    DS4G_K_P_SHARED_DOWN = 21,/* shared expert down GEMM + residual */
    DS4G_K_P_COMBINE = 22,    /* slot-order combine + the next layer's RMSNorm */
    DS4G_K_COUNT = 23
};
int ds4g_session_set_timing(ds4g_session *s, int on);

/* Tracing of the single-launch decode step: when buf (device, caller-owned) is
 * not NULL, each later decode step writes the GPU global time (ns) at which every
 * CTA starts each stage: entry [e * n_cta + c] for event e = 7 * layer + stage
 * (stages: Q/KV down, up + RoPE + append, attention, output projection, router,
 * gate/up, down + combine), e = 7 * n_layers for the lm_head and 7 * n_layers + 1
 * for the end; n_cta is the number of SMs.  Events beyond bytes / (8 n_cta) are
 * dropped.  NULL turns tracing off. */
int ds4g_session_set_trace(ds4g_session *s, void *buf, size_t bytes);
int ds4g_session_timing(ds4g_session *s, double *ms, uint64_t *counts, int n);

/* Sampler workspace bytes for a vocabulary of n_vocab (device memory). */
size_t ds4g_sample_workspace_bytes(int n_vocab);

/* [P3] 阶段四 4.3 sample_full_vocab.  logits: device f32 [n_vocab].
 * temperature <= 0: argmax, lowest id on ties; rng_state untouched.
 * temperature > 0: z = logits / T, p = exp(z - max z); top-p keeps the most
 * probable tokens (ties to the lower id) until their sum reaches top_p of the
 * total (top_p >= 1 keeps all); one draw u = (xorshift64*(rng_state) >> 40) / 2^24
 * advances *rng_state (host, nonzero); the result is the first token, in
 * vocabulary order, at which the running sum of kept probabilities reaches
 * u * (their total).  Probabilities are summed exactly in 2^-40 fixed point, so
 * the result does not depend on the order of device reductions.
 * workspace: device, >= ds4g_sample_workspace_bytes(n_vocab) bytes, 256-byte
 * aligned.  Synchronises `cuda_stream`. */
int32_t ds4g_sample(const float *logits, int n_vocab, float temperature, float top_p,
                    uint64_t *rng_state, void *workspace, size_t workspace_bytes,
                    void *cuda_stream);

/* As ds4g_sample with the uniform draw given by the caller: u = u24 / 2^24,
 * u24 < 2^24 (else DS4G_EINVAL); no RNG state is used.  For callers that bring
 * their own random numbers. */
int32_t ds4g_sample_u(const float *logits, int n_vocab, float temperature, float top_p,
                      uint32_t u24, void *workspace, size_t workspace_bytes, void *cuda_stream);

/* [P3] 阶段四 sample_top_p_min_p (named there with top-p, without a definition):
 * ds4g_sample with a min-p filter as well.  Reading: of the top-p set, a token is
 * kept only if its probability is at least min_p times the largest probability;
 * min_p = 0 is ds4g_sample, min_p = 1 keeps the most probable token (and its exact
 * ties).  0 <= min_p <= 1, else DS4G_EINVAL.  Everything else as ds4g_sample. */
int32_t ds4g_sample_min_p(const float *logits, int n_vocab, float temperature, float top_p, float min_p,
                          uint64_t *rng_state, void *workspace, size_t workspace_bytes,
                          void *cuda_stream);
/* ds4g_sample_min_p with the uniform draw given by the caller, as ds4g_sample_u. */
int32_t ds4g_sample_u_min_p(const float *logits, int n_vocab, float temperature, float top_p, float min_p,
                            uint32_t u24, void *workspace, size_t workspace_bytes, void *cuda_stream);

/* Largest vocabulary ds4g_sample_static accepts. */
#define DS4G_SAMPLE_STATIC_MAX_VOCAB 262144

/* ds4g_sample without a caller workspace.  The pages have no counterpart: this is
 * a library convenience.  It is for callers that cannot allocate device memory
 * for a workspace: a host program that only holds a logits pointer produced by
 * another library (it owns no device allocator), or a decode loop that must not
 * call cudaMalloc between steps, because cudaMalloc can synchronise the device.
 * Its scratch is a fixed 16 KB array in the library's device image, which exists
 * once the module is loaded; the call allocates nothing.  n_vocab above
 * DS4G_SAMPLE_STATIC_MAX_VOCAB returns DS4G_ESIZE; other arguments and the result
 * are as for ds4g_sample.  Every call looks up the scratch's address on the
 * current device (cudaGetSymbolAddress, which allocates nothing), so a device reset
 * between calls is safe.  There is one scratch per device: calls that overlap in
 * time on one device (two host threads, or two streams whose calls are not
 * ordered) race on it and give undefined results.  The scratch keeps the last
 * call's contents; each call clears the part that must start at zero.
 * Synchronises `cuda_stream`. */
int32_t ds4g_sample_static(const float *logits, int n_vocab, float temperature, float top_p,
                           uint64_t *rng_state, void *cuda_stream);

const char *ds4g_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* DS4G_H */
