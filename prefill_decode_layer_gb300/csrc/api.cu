// C ABI of the ds4g library (include/ds4g.h): model and session bookkeeping,
// validation, and the order in which the kernels of a call are issued.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <new>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "prefill_tc.h"

using namespace ds4g;

struct ds4g_model {
    ds4g_config cfg;
    Dims d;
    std::vector<LayerPtrs> layers;
    const uint16_t *tok_embd;
    const void *lm_head;
    int nsm;
    bool persistent;   // decode steps use the single cooperative launch
    bool tc;           // prefill GEMMs run on the tensor cores
    bool hilo;         // ... with every activation as a BF16 hi/lo pair
    std::vector<TcLayerMaps> tcmaps;   // per layer, when tc
};

struct ds4g_session {
    ds4g_model *m;
    int n_ctx;
    int len;
    std::vector<int32_t> hist;
    cudaStream_t st;
    std::vector<void *> kc, vc;
    float2 *rope;
    DecodeBufs b;
    PrefillBufs pb;
    TcActMaps tcact;            // tensor maps of pb's activations, when the model's prefill is tc
    std::vector<TcKVMaps> tckv; // per-layer K/V cache maps of the tcgen05 attention (when eligible)
    LayerPtrs *layers_dev;      // [L] device copy of the layer table
    void **kv_dev;              // [2L] device K then V cache pointers
    unsigned *bar;              // grid-barrier arrival counter of the persistent kernel
    unsigned bar_count = 0;     // its value after every launch so far (host copy)
    unsigned kv_count = 0;      // K/V-row counter (bar[1]) after every launch so far
    unsigned *qflag;            // [NH] per-head query-half flags of the persistent kernel
    unsigned q_count = 0;       // their value after every launch so far
    int *status;                // device status word
    std::vector<void *> kv_host;
    uint64_t launches = 0;
    unsigned long long *trace = nullptr;
    int trace_events = 0;
    float *last_x = nullptr;          // [L+1][H] layer inputs of the last prefilled token
    std::vector<int32_t> probe_pos;   // positions whose layer inputs are recorded
    float *probe_buf = nullptr;       // caller's [n][L+1][H] record buffer
    unsigned *done_h = nullptr;       // pinned host word the persistent kernel signals through
    unsigned *done_d = nullptr;       // its device view
    unsigned done_seq = 0;            // value of the last signal asked for
    bool timing = false;
    cudaEvent_t ev[DS4G_K_COUNT][2];
    PrefillBufs::Timing *ptm = nullptr;   // timing mode: the prefill's event chain
    double t_ms[DS4G_K_COUNT] = {};
    uint64_t t_n[DS4G_K_COUNT] = {};
};

namespace {
// Adds the kernels launched on this thread during a call to the session's count.
struct LaunchScope {
    ds4g_session *s;
    uint64_t start;
    explicit LaunchScope(ds4g_session *s_) : s(s_), start(ds4g::launch_count()) {}
    ~LaunchScope() { s->launches += ds4g::launch_count() - start; }
};
}  // namespace

namespace {

size_t al(size_t x) { return (x + 255) & ~(size_t)255; }

int prefill_P(const ds4g_config &c) { return c.prefill_chunk > 0 ? c.prefill_chunk : 4096; }

Dims dims_of(const ds4g_config &c)
{
    Dims d;
    d.L = c.n_layers; d.H = c.hidden; d.NH = c.n_heads; d.HD = c.head_dim; d.RQ = c.q_rank;
    d.RKV = c.kv_rank; d.W = c.window; d.E = c.n_experts; d.K = c.top_k; d.I = c.expert_inter;
    d.V = c.vocab; d.QD = c.n_heads * c.head_dim; d.eps = c.rms_eps; d.wdt = c.weight_dtype;
    d.kvdt = c.kv_dtype;
    return d;
}

bool cfg_ok(const ds4g_config *c)
{
    if (!c) return false;
    if (c->n_layers < 1 || c->hidden < 8 || c->n_heads < 1 || c->head_dim < 8) return false;
    if (c->hidden % 8 || c->q_rank % 8 || c->kv_rank % 8 || c->expert_inter % 8) return false;
    if (c->head_dim % 8 || c->head_dim > 256 || c->q_rank < 8 || c->kv_rank < 8) return false;
    if (c->window < 1 || c->window > 1024) return false;
    if (c->n_experts < 1 || c->n_experts > 1024 || c->top_k < 1 || c->top_k > 8 ||
        c->top_k > c->n_experts)
        return false;
    if (c->vocab < 1 || c->expert_inter < 8) return false;
    if (c->weight_dtype != DS4G_F32 && c->weight_dtype != DS4G_BF16) return false;
    if (c->kv_dtype != DS4G_F32 && c->kv_dtype != DS4G_BF16) return false;
    if (c->prefill_chunk < 0 || c->prefill_chunk > 65536) return false;
    if (c->decode_kernel != DS4G_DECODE_AUTO && c->decode_kernel != DS4G_DECODE_STAGED) return false;
    if (c->prefill_kernel != DS4G_PREFILL_AUTO && c->prefill_kernel != DS4G_PREFILL_SIMT &&
        c->prefill_kernel != DS4G_PREFILL_HILO)
        return false;
    if (!(c->rope_base > 0.f) || !(c->rms_eps >= 0.f)) return false;
    if (c->n_experts % 4) return false;  // 4-wide epilogues of the batched kernels
    // shared-memory footprints of the kernels (floats unless stated)
    const size_t smem_max = 227 * 1024;
    const size_t kvs = c->kv_dtype == DS4G_BF16 ? 2 : 4;
    const size_t win = 2 * (size_t)c->window * c->head_dim * kvs;
    if (win + (size_t)(c->head_dim + c->window + 32) * 4 > smem_max) return false;
    if (win + 8 * (size_t)(c->head_dim + c->window) * 4 > smem_max) return false;
    const size_t qd = (size_t)c->n_heads * c->head_dim;
    const size_t vecs[] = {(size_t)(c->hidden > c->n_experts ? c->hidden : c->n_experts) + 32,
                           (size_t)c->q_rank + c->kv_rank, qd,
                           (size_t)(c->top_k + 1) * c->expert_inter};
    for (size_t v : vecs)
        if (v * 4 > smem_max) return false;
    return true;
}

bool aligned16(const void *p) { return p && ((uintptr_t)p & 15u) == 0; }

struct Layout {
    size_t kv, rope, dec, pre, total;
};

Layout layout(const ds4g_config &c, int n_ctx)
{
    const Dims d = dims_of(c);
    const size_t kvs = c.kv_dtype == DS4G_BF16 ? 2 : 4;
    Layout L;
    size_t o = 0;
    L.kv = o;
    o += (size_t)d.L * 2 * al((size_t)n_ctx * d.HD * kvs);
    L.rope = o;
    o += al((size_t)n_ctx * (d.HD / 2) * sizeof(float2));
    L.dec = o;
    o += 4 * al((size_t)d.H * 4);                      // x, xm, xn2, hidden
    o += al((size_t)(d.RQ + d.RKV) * 4);               // c
    o += 2 * al((size_t)d.QD * 4);                     // q, o
    o += al((size_t)d.E * 4);                          // scores
    o += 2 * al((size_t)d.L * d.K * 4);                // ids, wts
    o += al((size_t)(d.K + 1) * d.I * 4);              // h
    o += al((size_t)d.V * 4);                          // logits
    o += al(64);                                       // counters
    o += al(64);                                       // barrier + status
    o += al((size_t)d.NH * 4);                         // per-head query-half flags
    o += al((size_t)d.L * sizeof(LayerPtrs));          // layer table
    o += al((size_t)2 * d.L * sizeof(void *));         // K/V pointer table
    o += al((size_t)(d.L + 1) * d.H * 4);              // prefill: last token entering each layer
    L.pre = o;
    o += prefill_bytes(d, prefill_P(c));
    L.total = o;
    return L;
}

__global__ void k_rope_table(float2 *t, int n_ctx, int half, double base)
{
    const size_t total = (size_t)n_ctx * half;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const int p = (int)(i / half), j = (int)(i % half);
        const double theta = pow(base, -2.0 * (double)j / (double)(2 * half));
        double s, c;
        sincos((double)p * theta, &s, &c);
        t[i] = make_float2((float)c, (float)s);
    }
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? DS4G_OK : DS4G_ECUDA; }

// xorshift64* (Vigna 2016): shifts 12, 25, 27; output multiplied by the published constant.
uint64_t xorshift64s(uint64_t *s)
{
    uint64_t x = *s;
    x ^= x >> 12;
    x ^= x << 25;
    x ^= x >> 27;
    *s = x;
    return x * 0x2545F4914F6CDD1DULL;
}

StepArgs step_base(ds4g_session *s)
{
    StepArgs a;
    memset(&a, 0, sizeof(a));
    a.d = s->m->d;
    a.rope = s->rope;
    a.b = s->b;
    a.tok_embd = s->m->tok_embd;
    a.lm_head = s->m->lm_head;
    a.token = -1;
    return a;
}

}  // namespace

extern "C" {

int ds4g_model_create(const ds4g_config *cfg, const ds4g_weights *w, ds4g_model **out)
{
    if (!out) return DS4G_EINVAL;
    *out = nullptr;
    if (!cfg_ok(cfg) || !w || !w->layers) return DS4G_EINVAL;
    if (!aligned16(w->tok_embd) || !aligned16(w->lm_head)) return DS4G_EINVAL;
    ds4g_model *m = new (std::nothrow) ds4g_model;
    if (!m) return DS4G_EINVAL;
    m->cfg = *cfg;
    m->d = dims_of(*cfg);
    m->tok_embd = static_cast<const uint16_t *>(w->tok_embd);
    m->lm_head = w->lm_head;
    for (int l = 0; l < cfg->n_layers; ++l) {
        const ds4g_layer_weights &s = w->layers[l];
        const void *all[] = {s.attn_norm, s.wq_a, s.wq_b, s.wkv_a, s.wk_b, s.wv_b, s.wo,
                             s.ffn_norm, s.w_router, s.w_gate, s.w_up, s.w_down, s.ws_gate,
                             s.ws_up, s.ws_down};
        for (const void *p : all)
            if (!aligned16(p)) { delete m; return DS4G_EINVAL; }
        LayerPtrs L;
        L.attn_norm = static_cast<const float *>(s.attn_norm);
        L.wq_a = s.wq_a; L.wq_b = s.wq_b; L.wkv_a = s.wkv_a; L.wk_b = s.wk_b; L.wv_b = s.wv_b;
        L.wo = s.wo;
        L.ffn_norm = static_cast<const float *>(s.ffn_norm);
        L.w_router = s.w_router; L.w_gate = s.w_gate; L.w_up = s.w_up; L.w_down = s.w_down;
        L.ws_gate = s.ws_gate; L.ws_up = s.ws_up; L.ws_down = s.ws_down;
        m->layers.push_back(L);
    }
    int dev = 0, max_smem = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (!e) e = cudaDeviceGetAttribute(&m->nsm, cudaDevAttrMultiProcessorCount, dev);
    if (!e) e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (!e) e = decode_setup(m->d, max_smem);
    if (!e) e = prefill_setup(m->d, max_smem);
    m->persistent = false;
    if (!e && cfg->decode_kernel == DS4G_DECODE_AUTO)
        e = persistent_setup(m->d, max_smem, m->nsm, &m->persistent);
    m->tc = !e && (cfg->prefill_kernel == DS4G_PREFILL_AUTO || cfg->prefill_kernel == DS4G_PREFILL_HILO) &&
            tc_prefill_eligible(m->d);
    m->hilo = cfg->prefill_kernel == DS4G_PREFILL_HILO;
    if (m->tc) {
        e = attn_mma_setup(m->d, max_smem);
        if (!e) e = attn_tc_setup(m->d, max_smem);
        m->tcmaps.resize(m->layers.size());
        for (size_t l = 0; !e && l < m->layers.size(); ++l) e = tc_layer_maps(m->d, m->layers[l], m->tcmaps[l]);
    }
    if (e) {
        if (getenv("DS4G_VERBOSE")) fprintf(stderr, "ds4g_model_create: %s\n", cudaGetErrorString(e));
        delete m;
        return DS4G_ECUDA;
    }
    *out = m;
    return DS4G_OK;
}

void ds4g_model_destroy(ds4g_model *m) { delete m; }

size_t ds4g_session_bytes(const ds4g_config *cfg, int n_ctx)
{
    if (!cfg_ok(cfg) || n_ctx < 1) return 0;
    return layout(*cfg, n_ctx).total;
}

static void destroy_side(PrefillBufs &pb)
{
    if (pb.ev_fork) cudaEventDestroy(pb.ev_fork);
    if (pb.ev_join) cudaEventDestroy(pb.ev_join);
    if (pb.side) cudaStreamDestroy(pb.side);
    pb.side = nullptr;
    pb.ev_fork = pb.ev_join = nullptr;
}

int ds4g_session_create(ds4g_model *m, int n_ctx, void *dev_mem, size_t bytes, void *stream,
                        ds4g_session **out)
{
    if (!out) return DS4G_EINVAL;
    *out = nullptr;
    if (!m || n_ctx < 1 || !dev_mem || ((uintptr_t)dev_mem & 255u)) return DS4G_EINVAL;
    const Layout L = layout(m->cfg, n_ctx);
    if (bytes < L.total) return DS4G_ESIZE;
    ds4g_session *s = new (std::nothrow) ds4g_session;
    if (!s) return DS4G_EINVAL;
    const Dims &d = m->d;
    char *base = static_cast<char *>(dev_mem);
    s->m = m;
    s->n_ctx = n_ctx;
    s->len = 0;
    s->hist.assign((size_t)n_ctx, 0);
    s->st = static_cast<cudaStream_t>(stream);
    if (m->tc &&
        (cudaStreamCreateWithFlags(&s->pb.side, cudaStreamNonBlocking) ||
         cudaEventCreateWithFlags(&s->pb.ev_fork, cudaEventDisableTiming) ||
         cudaEventCreateWithFlags(&s->pb.ev_join, cudaEventDisableTiming))) {
        destroy_side(s->pb);
        delete s;
        return DS4G_ECUDA;
    }
    const size_t kvs = m->cfg.kv_dtype == DS4G_BF16 ? 2 : 4;
    const size_t per = al((size_t)n_ctx * d.HD * kvs);
    for (int l = 0; l < d.L; ++l) {
        s->kc.push_back(base + L.kv + (2 * (size_t)l) * per);
        s->vc.push_back(base + L.kv + (2 * (size_t)l + 1) * per);
    }
    s->rope = reinterpret_cast<float2 *>(base + L.rope);
    char *p = base + L.dec;
    auto take = [&](size_t n) { char *r = p; p += al(n); return r; };
    DecodeBufs &b = s->b;
    b.x = (float *)take((size_t)d.H * 4);
    b.xm = (float *)take((size_t)d.H * 4);
    b.xn2 = (float *)take((size_t)d.H * 4);
    b.hidden = (float *)take((size_t)d.H * 4);
    b.c = (float *)take((size_t)(d.RQ + d.RKV) * 4);
    b.q = (float *)take((size_t)d.QD * 4);
    b.o = (float *)take((size_t)d.QD * 4);
    b.scores = (float *)take((size_t)d.E * 4);
    b.ids = (int *)take((size_t)d.L * d.K * 4);
    b.wts = (float *)take((size_t)d.L * d.K * 4);
    b.h = (float *)take((size_t)(d.K + 1) * d.I * 4);
    b.logits = (float *)take((size_t)d.V * 4);
    b.counters = (unsigned *)take(64);
    b.layer_x = nullptr;
    b.x_out = nullptr;
    s->bar = (unsigned *)take(64);
    s->status = (int *)(s->bar + 4);
    s->qflag = (unsigned *)take((size_t)d.NH * 4);
    b.status = s->status;
    s->layers_dev = (LayerPtrs *)take((size_t)d.L * sizeof(LayerPtrs));
    s->kv_dev = (void **)take((size_t)2 * d.L * sizeof(void *));
    float *layer_x = (float *)take((size_t)(d.L + 1) * d.H * 4);
    s->kv_host.assign(s->kc.begin(), s->kc.end());
    s->kv_host.insert(s->kv_host.end(), s->vc.begin(), s->vc.end());
    prefill_carve(d, prefill_P(m->cfg), base + L.pre, s->pb);
    s->pb.status = s->status;
    s->pb.n_rec = 0;
    s->last_x = layer_x;
    if (m->tc && tc_act_maps(d, s->pb, s->tcact)) {
        delete s;
        return DS4G_ECUDA;
    }
    if (m->tc && attn_tc_eligible(d)) {
        s->tckv.resize(d.L);
        for (int l = 0; l < d.L; ++l)
            if (attn_tc_kv_maps(d, s->kc[l], s->vc[l], n_ctx, s->tckv[l])) {
                delete s;
                return DS4G_ECUDA;
            }
    }
    cudaError_t e = cudaMemsetAsync(base + L.dec, 0, L.pre - L.dec, s->st);
    if (!e) e = cudaMemcpyAsync(s->layers_dev, m->layers.data(), (size_t)d.L * sizeof(LayerPtrs),
                                cudaMemcpyHostToDevice, s->st);
    if (!e) e = cudaMemcpyAsync(s->kv_dev, s->kv_host.data(), (size_t)2 * d.L * sizeof(void *),
                                cudaMemcpyHostToDevice, s->st);
    if (!e) e = cudaStreamSynchronize(s->st);  // the host tables above are read by the copies
    if (!e) {
        k_rope_table<<<256, 256, 0, s->st>>>(s->rope, n_ctx, d.HD / 2, (double)m->cfg.rope_base);
        ++launch_count();
        e = cudaGetLastError();
    }
    if (e) { delete s; return DS4G_ECUDA; }
    *out = s;
    return DS4G_OK;
}

void ds4g_session_destroy(ds4g_session *s)
{
    if (!s) return;
    if (s->done_h) cudaFreeHost(s->done_h);
    if (s->pb.side) cudaStreamSynchronize(s->pb.side);
    destroy_side(s->pb);
    if (s->timing) {
        cudaStreamSynchronize(s->st);
        for (int k = 0; k < DS4G_K_COUNT; ++k) {
            cudaEventDestroy(s->ev[k][0]);
            cudaEventDestroy(s->ev[k][1]);
        }
        for (int i = 0; i < PrefillBufs::Timing::kMax; ++i) cudaEventDestroy(s->ptm->ev[i]);
        delete s->ptm;
    }
    delete s;
}

int ds4g_prefill(ds4g_session *s, const int32_t *tokens, int n)
{
    if (!s || n < 0 || (n > 0 && !tokens)) return DS4G_EINVAL;
    if (n == 0) return DS4G_OK;
    const Dims &d = s->m->d;
    for (int i = 0; i < n; ++i)
        if (tokens[i] < 0 || tokens[i] >= d.V) return DS4G_ETOKEN;
    if ((long long)s->len + n >= s->n_ctx) return DS4G_ECONTEXT;
    LaunchScope scope(s);
    const int P = s->pb.P;
    for (int c = 0; c < n; c += P) {
        const int nc = n - c < P ? n - c : P;
        // record the last token's layer inputs, and those of probed positions in this chunk
        s->pb.n_rec = 0;
        if (c + nc == n) {
            s->pb.rec_row[0] = nc - 1;
            s->pb.rec_dst[0] = s->last_x;
            s->pb.n_rec = 1;
        }
        if (s->probe_buf)
            for (size_t i = 0; i < s->probe_pos.size(); ++i) {
                const int r = s->probe_pos[i] - (s->len + c);
                if (r < 0 || r >= nc) continue;
                s->pb.rec_row[s->pb.n_rec] = r;
                s->pb.rec_dst[s->pb.n_rec] = s->probe_buf + i * (size_t)(d.L + 1) * d.H;
                ++s->pb.n_rec;
            }
        cudaError_t e = cudaMemcpyAsync(s->pb.tok, tokens + c, (size_t)nc * 4,
                                        cudaMemcpyHostToDevice, s->st);
        if (!e)
            e = s->m->tc ? prefill_chunk_tc(d, s->m->layers.data(), s->m->tcmaps.data(), s->tcact,
                                            s->tckv.empty() ? nullptr : s->tckv.data(), s->kc.data(),
                                            s->vc.data(), s->rope, s->m->tok_embd, s->pb, s->len + c, nc, s->st,
                                            s->m->nsm, s->m->hilo)
                         : prefill_chunk(d, s->m->layers.data(), s->kc.data(), s->vc.data(), s->rope,
                                         s->m->tok_embd, s->pb, s->len + c, nc, s->st, s->m->nsm);
        if (!e && s->ptm && s->ptm->n > 0) {   // timing mode: each launch's share of the chunk
            PrefillBufs::Timing &tm = *s->ptm;
            e = cudaEventSynchronize(tm.ev[tm.n - 1]);
            for (int i = 1; !e && i < tm.n; ++i) {
                float ms = 0.f;
                e = cudaEventElapsedTime(&ms, tm.ev[i - 1], tm.ev[i]);
                if (!e && tm.kind[i] >= 0 && tm.kind[i] < DS4G_K_COUNT) {
                    s->t_ms[tm.kind[i]] += ms;
                    s->t_n[tm.kind[i]] += 1;
                }
            }
            tm.n = 0;
        }
        if (!e && c + nc == n) {  // last token's hidden state, then its logits
            e = cudaMemcpyAsync(s->b.x, s->pb.X + (size_t)(nc - 1) * d.H, (size_t)d.H * 4,
                                cudaMemcpyDeviceToDevice, s->st);
            if (!e) e = decode_lm_head(step_base(s), s->st, s->m->nsm);
        }
        if (e) return DS4G_ECUDA;
    }
    memcpy(s->hist.data() + s->len, tokens, (size_t)n * 4);
    s->len += n;
    return DS4G_OK;
}

// Where a persistent launch hands its result to a waiting host thread: the final
// hidden state into x_out (a device view of pinned host memory) and a completion
// signal into the session's pinned word.  `used` tells whether the launch took it.
struct HostOut {
    float *x_out = nullptr;
    bool used = false;
};

static int decode_common(ds4g_session *s, int32_t token, bool logits, HostOut *ho = nullptr)
{
    if (!s) return DS4G_EINVAL;
    const Dims &d = s->m->d;
    if (token < 0 || token >= d.V) return DS4G_ETOKEN;
    if (s->len + 1 >= s->n_ctx) return DS4G_ECONTEXT;
    LaunchScope scope(s);
    float *rec = nullptr;   // layer inputs of this position, when it is probed
    if (s->probe_buf)
        for (size_t i = 0; i < s->probe_pos.size(); ++i)
            if (s->probe_pos[i] == s->len) rec = s->probe_buf + i * (size_t)(d.L + 1) * d.H;
    if (s->m->persistent && !s->timing) {
        PersistArgs pa;
        memset(&pa, 0, sizeof(pa));
        pa.d = d;
        pa.layers = s->layers_dev;
        pa.kc = s->kv_dev;
        pa.vc = s->kv_dev + d.L;
        pa.rope = s->rope;
        pa.b = s->b;
        pa.b.layer_x = rec;
        if (ho && s->done_d) {
            pa.b.x_out = ho->x_out;
            if (++s->done_seq == 0) s->done_seq = 1;   // 0 is the word's initial value
            pa.done_flag = s->done_d;
            pa.done_seq = s->done_seq;
        }
        pa.tok_embd = s->m->tok_embd;
        pa.lm_head = s->m->lm_head;
        pa.pos = s->len;
        pa.token = token;
        pa.logits = logits ? 1 : 0;
        pa.bar = s->bar;
        pa.bar_base = s->bar_count;
        pa.kv_base = s->kv_count;
        pa.qflag = s->qflag;
        pa.q_base = s->q_count;
        pa.split_q = 2 * d.NH + 2 <= s->m->nsm;
        pa.status = s->status;
        pa.trace = s->trace;
        pa.trace_events = s->trace_events;
        if (decode_persistent(pa, s->st, s->m->nsm)) return DS4G_ECUDA;
        // grid barriers per launch: five inside every layer, one between layers and
        // one before the lm_head; two K/V-row publications per layer
        s->bar_count += (unsigned)(6 * d.L - 1 + pa.logits) * (unsigned)s->m->nsm;
        s->kv_count += 2u * (unsigned)d.L;
        if (pa.split_q) s->q_count += (unsigned)d.L;   // one query half per head and layer
        s->hist[s->len] = token;
        s->len += 1;
        if (ho) ho->used = pa.done_flag != nullptr;
        return DS4G_OK;
    }
    StepArgs a = step_base(s);
    a.pos = s->len;
    a.b.layer_x = rec;   // row 0 (the embedding) is written by the first kernel
    cudaEvent_t(*ev)[2] = s->timing ? s->ev : nullptr;
    for (int l = 0; l < d.L; ++l) {
        a.w = s->m->layers[l];
        a.kc = s->kc[l];
        a.vc = s->vc[l];
        a.layer = l;
        a.token = l == 0 ? token : -1;
        if (decode_layer(a, s->st, s->m->nsm, ev)) return DS4G_ECUDA;
        if (rec && cudaMemcpyAsync(rec + (size_t)(l + 1) * d.H, s->b.x, (size_t)d.H * 4,
                                   cudaMemcpyDeviceToDevice, s->st))
            return DS4G_ECUDA;
        if (ev) {  // read this layer's kernel times before the events are reused
            if (cudaStreamSynchronize(s->st)) return DS4G_ECUDA;
            for (int k = 0; k <= DS4G_K_EXPERT_DOWN; ++k) {
                float ms = 0.f;
                if (cudaEventElapsedTime(&ms, ev[k][0], ev[k][1])) return DS4G_ECUDA;
                s->t_ms[k] += ms;
                s->t_n[k] += 1;
            }
        }
    }
    a.token = -1;
    if (!logits) {
        s->hist[s->len] = token;
        s->len += 1;
        return DS4G_OK;
    }
    if (ev) cudaEventRecord(ev[DS4G_K_LM_HEAD][0], s->st);
    if (decode_lm_head(a, s->st, s->m->nsm)) return DS4G_ECUDA;
    if (ev) {
        float ms = 0.f;
        cudaEventRecord(ev[DS4G_K_LM_HEAD][1], s->st);
        if (cudaEventSynchronize(ev[DS4G_K_LM_HEAD][1]) ||
            cudaEventElapsedTime(&ms, ev[DS4G_K_LM_HEAD][0], ev[DS4G_K_LM_HEAD][1]))
            return DS4G_ECUDA;
        s->t_ms[DS4G_K_LM_HEAD] += ms;
        s->t_n[DS4G_K_LM_HEAD] += 1;
    }
    s->hist[s->len] = token;
    s->len += 1;
    return DS4G_OK;
}

int ds4g_decode_step(ds4g_session *s, int32_t token) { return decode_common(s, token, true); }

int ds4g_decode_layers(ds4g_session *s, int32_t token) { return decode_common(s, token, false); }

// The session's pinned completion word (allocated on first use; host memory).
static bool done_word(ds4g_session *s)
{
    if (s->done_h) return true;
    void *h = nullptr, *dv = nullptr;
    if (cudaHostAlloc(&h, 64, cudaHostAllocMapped) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (cudaHostGetDevicePointer(&dv, h, 0) != cudaSuccess) {
        cudaGetLastError();
        cudaFreeHost(h);
        return false;
    }
    s->done_h = static_cast<unsigned *>(h);
    s->done_d = static_cast<unsigned *>(dv);
    __atomic_store_n(s->done_h, 0u, __ATOMIC_RELEASE);
    return true;
}

// Waits for the launch's completion signal.  Every wait inside the kernel is
// bounded, so the stream drains in any case; a drained stream without the signal
// means the kernel gave up (DS4G_ETIMEOUT), and the ticket is cleared for the next
// launch.
static int wait_done(ds4g_session *s, unsigned seq)
{
    for (unsigned n = 1;; ++n) {
        if (__atomic_load_n(s->done_h, __ATOMIC_ACQUIRE) == seq) return DS4G_OK;
        if ((n & 255u) == 0) {
            const cudaError_t q = cudaStreamQuery(s->st);
            if (q == cudaErrorNotReady) continue;
            if (q != cudaSuccess) return cuda_status(q);
            if (__atomic_load_n(s->done_h, __ATOMIC_ACQUIRE) == seq) return DS4G_OK;
            cudaError_t e = cudaMemsetAsync(s->b.counters, 0, 64, s->st);
            if (!e) e = cudaStreamSynchronize(s->st);
            return e ? cuda_status(e) : DS4G_ETIMEOUT;
        }
    }
}

int ds4g_decode_layers_host(ds4g_session *s, int32_t token, float *hidden_host)
{
    if (!s || !hidden_host) return DS4G_EINVAL;
    // Pinned (page-locked) host memory has a device view: the persistent kernel writes
    // the hidden state there itself and signals completion through a pinned word, so
    // the step needs neither a copy-engine transfer nor a stream synchronisation.
    // Other memory gets the copy.
    HostOut ho;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, hidden_host) == cudaSuccess) {
        if (at.type == cudaMemoryTypeHost && at.devicePointer && done_word(s))   // dereferenceable here
            ho.x_out = static_cast<float *>(at.devicePointer);
    } else {
        cudaGetLastError();   // not a pointer the runtime knows: plain host memory
    }
    const int rc = decode_common(s, token, false, ho.x_out ? &ho : nullptr);
    if (rc) return rc;
    if (ho.used) return wait_done(s, s->done_seq);
    cudaError_t e = cudaMemcpyAsync(hidden_host, s->b.x, (size_t)s->m->d.H * 4, cudaMemcpyDeviceToHost, s->st);
    if (!e) e = cudaStreamSynchronize(s->st);
    return cuda_status(e);
}

int ds4g_session_common_prefix(const ds4g_session *s, const int32_t *tokens, int n)
{
    if (!s || n < 0 || (n > 0 && !tokens)) return DS4G_EINVAL;
    int i = 0;
    while (i < n && i < s->len && s->hist[i] == tokens[i]) ++i;
    return i;
}

int ds4g_session_truncate(ds4g_session *s, int common_prefix)
{
    if (!s || common_prefix < 0 || common_prefix > s->len) return DS4G_EINVAL;
    s->len = common_prefix;
    return DS4G_OK;
}

// Checks of a prompt that come before a sync or a rewrite changes the session.
static int prompt_ok(const ds4g_session *s, const int32_t *tokens, int n)
{
    if (!s || n < 0 || (n > 0 && !tokens)) return DS4G_EINVAL;
    if (n >= s->n_ctx) return DS4G_ECONTEXT;
    for (int i = 0; i < n; ++i)
        if (tokens[i] < 0 || tokens[i] >= s->m->d.V) return DS4G_ETOKEN;
    return DS4G_OK;
}

int ds4g_session_sync(ds4g_session *s, const int32_t *tokens, int n, int *n_prefilled)
{
    if (n_prefilled) *n_prefilled = 0;
    const int rc = prompt_ok(s, tokens, n);
    if (rc) return rc;
    int cp = ds4g_session_common_prefix(s, tokens, n);
    if (cp == n && n > 0) cp = n - 1;   // its logits are gone: run the last token again
    s->len = cp;
    if (n == cp) return DS4G_OK;
    const int e = ds4g_prefill(s, tokens + cp, n - cp);
    if (e == DS4G_OK && n_prefilled) *n_prefilled = n - cp;
    return e;
}

int ds4g_session_rewrite_from_common(ds4g_session *s, const int32_t *tokens, int n, int common)
{
    const int rc = prompt_ok(s, tokens, n);
    if (rc) return rc;
    if (common < 0 || common > ds4g_session_common_prefix(s, tokens, n)) return DS4G_EINVAL;
    if (common == n && n == s->len) return DS4G_OK;   // the checkpoint already holds the prompt
    s->len = common;
    return n > common ? ds4g_prefill(s, tokens + common, n - common) : DS4G_OK;
}

int ds4g_session_len(const ds4g_session *s) { return s ? s->len : DS4G_EINVAL; }

const float *ds4g_session_logits(const ds4g_session *s) { return s ? s->b.logits : nullptr; }

const float *ds4g_session_hidden(const ds4g_session *s) { return s ? s->b.x : nullptr; }

int ds4g_session_kv(ds4g_session *s, int layer, void **k, void **v)
{
    if (!s || layer < 0 || layer >= s->m->d.L || !k || !v) return DS4G_EINVAL;
    *k = s->kc[layer];
    *v = s->vc[layer];
    return DS4G_OK;
}

int ds4g_session_restore(ds4g_session *s, const int32_t *tokens, int n)
{
    if (!s || n < 0 || (n > 0 && !tokens)) return DS4G_EINVAL;
    if (n >= s->n_ctx) return DS4G_ECONTEXT;
    for (int i = 0; i < n; ++i)
        if (tokens[i] < 0 || tokens[i] >= s->m->d.V) return DS4G_ETOKEN;
    if (n) memcpy(s->hist.data(), tokens, (size_t)n * 4);
    s->len = n;
    return DS4G_OK;
}

// ------------------------------------------------------------------ checkpoints
namespace {
struct CkptHeader {            // 64 bytes
    char magic[8];             // "DS4GKV01"
    uint32_t version, kv_size;
    int32_t n_layers, head_dim, n_tokens, reserved;
    uint64_t cfg_digest;
    uint8_t pad[24];
};
static_assert(sizeof(CkptHeader) == 64, "checkpoint header");
constexpr char kCkptMagic[8] = {'D', 'S', '4', 'G', 'K', 'V', '0', '1'};

// FNV-1a over the configuration fields that fix the cached state's meaning.
uint64_t cfg_digest(const ds4g_config &c)
{
    const int64_t f[] = {c.n_layers, c.hidden, c.n_heads, c.head_dim, c.q_rank, c.kv_rank, c.window,
                         c.n_experts, c.top_k, c.expert_inter, c.vocab, c.weight_dtype, c.kv_dtype};
    uint64_t h = 1469598103934665603ull;
    auto mix = [&](const void *p, size_t n) {
        const unsigned char *b = static_cast<const unsigned char *>(p);
        for (size_t i = 0; i < n; ++i) h = (h ^ b[i]) * 1099511628211ull;
    };
    mix(f, sizeof(f));
    mix(&c.rope_base, sizeof(c.rope_base));
    mix(&c.rms_eps, sizeof(c.rms_eps));
    return h;
}
size_t ckpt_tokens_bytes(int n) { return ((size_t)n * 4 + 15) & ~(size_t)15; }
size_t ckpt_rows_bytes(const ds4g_config &c, int n)
{
    return (size_t)n * c.head_dim * (c.kv_dtype == DS4G_BF16 ? 2 : 4);
}
}  // namespace

size_t ds4g_checkpoint_bytes(const ds4g_config *cfg, int n_tokens)
{
    if (!cfg_ok(cfg) || n_tokens < 0) return 0;
    return sizeof(CkptHeader) + ckpt_tokens_bytes(n_tokens) +
           (size_t)cfg->n_layers * 2 * ckpt_rows_bytes(*cfg, n_tokens);
}

int ds4g_session_save(ds4g_session *s, void *buf, size_t bytes)
{
    if (!s || !buf) return DS4G_EINVAL;
    const ds4g_config &c = s->m->cfg;
    const int n = s->len;
    if (bytes < ds4g_checkpoint_bytes(&c, n)) return DS4G_ESIZE;
    CkptHeader h;
    memset(&h, 0, sizeof(h));
    memcpy(h.magic, kCkptMagic, 8);
    h.version = 1;
    h.kv_size = c.kv_dtype == DS4G_BF16 ? 2 : 4;
    h.n_layers = c.n_layers;
    h.head_dim = c.head_dim;
    h.n_tokens = n;
    h.cfg_digest = cfg_digest(c);
    char *p = static_cast<char *>(buf);
    memcpy(p, &h, sizeof(h));
    p += sizeof(h);
    if (n) memcpy(p, s->hist.data(), (size_t)n * 4);
    p += ckpt_tokens_bytes(n);
    const size_t rows = ckpt_rows_bytes(c, n);
    cudaError_t e = cudaSuccess;
    for (int l = 0; !e && l < c.n_layers && rows; ++l) {
        e = cudaMemcpyAsync(p, s->kc[l], rows, cudaMemcpyDeviceToHost, s->st);
        p += rows;
        if (!e) e = cudaMemcpyAsync(p, s->vc[l], rows, cudaMemcpyDeviceToHost, s->st);
        p += rows;
    }
    if (!e) e = cudaStreamSynchronize(s->st);
    return cuda_status(e);
}

int ds4g_session_load(ds4g_session *s, const void *buf, size_t bytes)
{
    if (!s || !buf) return DS4G_EINVAL;
    const ds4g_config &c = s->m->cfg;
    if (bytes < sizeof(CkptHeader)) return DS4G_ESIZE;
    CkptHeader h;
    memcpy(&h, buf, sizeof(h));
    if (memcmp(h.magic, kCkptMagic, 8) || h.version != 1 || h.kv_size != (c.kv_dtype == DS4G_BF16 ? 2u : 4u) ||
        h.n_layers != c.n_layers || h.head_dim != c.head_dim || h.n_tokens < 0 || h.cfg_digest != cfg_digest(c))
        return DS4G_EINVAL;
    const int n = h.n_tokens;
    if (bytes < ds4g_checkpoint_bytes(&c, n)) return DS4G_ESIZE;
    if (n >= s->n_ctx) return DS4G_ECONTEXT;
    const char *p = static_cast<const char *>(buf) + sizeof(h);
    const int32_t *tok = reinterpret_cast<const int32_t *>(p);
    for (int i = 0; i < n; ++i)
        if (tok[i] < 0 || tok[i] >= s->m->d.V) return DS4G_ETOKEN;
    p += ckpt_tokens_bytes(n);
    const size_t rows = ckpt_rows_bytes(c, n);
    cudaError_t e = cudaSuccess;
    for (int l = 0; !e && l < c.n_layers && rows; ++l) {
        e = cudaMemcpyAsync(s->kc[l], p, rows, cudaMemcpyHostToDevice, s->st);
        p += rows;
        if (!e) e = cudaMemcpyAsync(s->vc[l], p, rows, cudaMemcpyHostToDevice, s->st);
        p += rows;
    }
    if (!e) e = cudaStreamSynchronize(s->st);
    if (e) {
        // Some layers' K/V rows may already be overwritten: the cache no longer
        // matches the history, so the session is emptied.
        s->len = 0;
        return cuda_status(e);
    }
    if (n) memcpy(s->hist.data(), tok, (size_t)n * 4);
    s->len = n;
    return DS4G_OK;
}

int ds4g_session_router(ds4g_session *s, int layer, int32_t *ids, float *weights)
{
    if (!s || layer < 0 || layer >= s->m->d.L || !ids || !weights) return DS4G_EINVAL;
    const int K = s->m->d.K;
    cudaError_t e = cudaMemcpyAsync(ids, s->b.ids + (size_t)layer * K, (size_t)K * 4,
                                    cudaMemcpyDeviceToHost, s->st);
    if (!e) e = cudaMemcpyAsync(weights, s->b.wts + (size_t)layer * K, (size_t)K * 4,
                                cudaMemcpyDeviceToHost, s->st);
    if (!e) e = cudaStreamSynchronize(s->st);
    return cuda_status(e);
}

const void *ds4g_session_debug(const ds4g_session *s, int which)
{
    if (!s) return nullptr;
    switch (which) {
    case DS4G_DBG_X: return s->b.x;
    case DS4G_DBG_CQKV: return s->b.c;
    case DS4G_DBG_Q: return s->b.q;
    case DS4G_DBG_ATTN: return s->b.o;
    case DS4G_DBG_XMID: return s->b.xm;
    case DS4G_DBG_XN2: return s->b.xn2;
    case DS4G_DBG_SCORES: return s->b.scores;
    case DS4G_DBG_H: return s->b.h;
    case DS4G_DBG_HIDDEN: return s->b.x;
    case DS4G_DBG_PREFILL_X: return s->pb.X;
    case DS4G_DBG_STATUS: return s->status;
    case DS4G_DBG_PREFILL_LAYER_X: return s->last_x;
    default: return nullptr;
    }
}

uint64_t ds4g_session_launches(const ds4g_session *s) { return s ? s->launches : 0; }

int ds4g_session_status(ds4g_session *s)
{
    if (!s) return DS4G_EINVAL;
    int st = 0;
    cudaError_t e = cudaMemcpyAsync(&st, s->status, 4, cudaMemcpyDeviceToHost, s->st);
    if (!e) e = cudaStreamSynchronize(s->st);
    if (e) return DS4G_ECUDA;
    if (st != 0) {  // clear the flag and the barrier counter a failed wait left behind
        e = cudaMemsetAsync(s->bar, 0, 64, s->st);
        if (!e) e = cudaMemsetAsync(s->qflag, 0, (size_t)s->m->d.NH * 4, s->st);
        if (!e) e = cudaStreamSynchronize(s->st);
        s->bar_count = 0;
        s->kv_count = 0;
        s->q_count = 0;
        if (e) return DS4G_ECUDA;
        return st == DS4G_ENONFINITE ? DS4G_ENONFINITE : DS4G_ETIMEOUT;
    }
    return DS4G_OK;
}

int ds4g_session_set_timing(ds4g_session *s, int on)
{
    if (!s) return DS4G_EINVAL;
    if (on && !s->timing) {
        // all events, or none (a failure destroys the ones already created)
        PrefillBufs::Timing *tm = new (std::nothrow) PrefillBufs::Timing();
        if (!tm) return DS4G_ECUDA;
        bool ok = true;
        int ke = 0;   // kinds whose two events exist
        for (; ke < DS4G_K_COUNT; ++ke) {
            if (cudaEventCreate(&s->ev[ke][0])) {
                ok = false;
                break;
            }
            if (cudaEventCreate(&s->ev[ke][1])) {
                cudaEventDestroy(s->ev[ke][0]);
                ok = false;
                break;
            }
        }
        int pe = 0;   // prefill events that exist
        for (; ok && pe < PrefillBufs::Timing::kMax; ++pe)
            if (cudaEventCreate(&tm->ev[pe])) {
                ok = false;
                break;
            }
        if (!ok) {
            for (int i = 0; i < pe; ++i) cudaEventDestroy(tm->ev[i]);
            for (int k = 0; k < ke; ++k) {
                cudaEventDestroy(s->ev[k][0]);
                cudaEventDestroy(s->ev[k][1]);
            }
            delete tm;
            return DS4G_ECUDA;
        }
        tm->n = 0;
        s->ptm = tm;
        s->pb.tm = tm;
        s->timing = true;
    } else if (!on && s->timing) {
        if (cudaStreamSynchronize(s->st)) return DS4G_ECUDA;
        for (int k = 0; k < DS4G_K_COUNT; ++k) {
            cudaEventDestroy(s->ev[k][0]);
            cudaEventDestroy(s->ev[k][1]);
        }
        s->pb.tm = nullptr;
        for (int i = 0; i < PrefillBufs::Timing::kMax; ++i) cudaEventDestroy(s->ptm->ev[i]);
        delete s->ptm;
        s->ptm = nullptr;
        s->timing = false;
    }
    return DS4G_OK;
}

int ds4g_session_set_probe(ds4g_session *s, const int32_t *positions, int n, float *buf)
{
    if (!s || n < 0 || n > kMaxProbe || (n > 0 && (!positions || !buf))) return DS4G_EINVAL;
    for (int i = 0; i < n; ++i)
        if (positions[i] < 0 || positions[i] >= s->n_ctx) return DS4G_EINVAL;
    s->probe_pos.assign(positions, positions + n);
    s->probe_buf = n > 0 ? buf : nullptr;
    return DS4G_OK;
}

int ds4g_session_set_trace(ds4g_session *s, void *buf, size_t bytes)
{
    if (!s) return DS4G_EINVAL;
    s->trace = static_cast<unsigned long long *>(buf);
    s->trace_events = buf ? (int)(bytes / (8 * (size_t)s->m->nsm)) : 0;
    return DS4G_OK;
}

int ds4g_session_timing(ds4g_session *s, double *ms, uint64_t *counts, int n)
{
    if (!s || n < 0 || (n > 0 && (!ms || !counts))) return DS4G_EINVAL;
    for (int k = 0; k < n && k < DS4G_K_COUNT; ++k) {
        ms[k] = s->t_ms[k];
        counts[k] = s->t_n[k];
    }
    for (int k = 0; k < DS4G_K_COUNT; ++k) {
        s->t_ms[k] = 0.0;
        s->t_n[k] = 0;
    }
    return DS4G_OK;
}

size_t ds4g_sample_workspace_bytes(int n_vocab)
{
    return n_vocab > 0 ? sample_workspace_bytes(n_vocab) : 0;
}

static int32_t sample_common(const float *logits, int n_vocab, float temperature, float top_p, float min_p,
                             unsigned u24, void *workspace, size_t workspace_bytes, void *stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int *res = nullptr;
    int32_t tok = -1;
    cudaError_t e = sample_launch(logits, n_vocab, temperature, top_p, min_p, u24, workspace, st, &res);
    if (!e) e = cudaMemcpyAsync(&tok, res, 4, cudaMemcpyDeviceToHost, st);
    if (!e) e = cudaStreamSynchronize(st);
    if (e) return DS4G_ECUDA;
    return tok;
}

static int sample_args_ok(const float *logits, int n_vocab, float temperature, float top_p,
                          void *workspace, size_t workspace_bytes)
{
    if (!logits || n_vocab < 1 || !workspace || ((uintptr_t)workspace & 255u)) return DS4G_EINVAL;
    if (workspace_bytes < sample_workspace_bytes(n_vocab)) return DS4G_ESIZE;
    if (temperature != temperature || top_p != top_p) return DS4G_EINVAL;
    return DS4G_OK;
}

int32_t ds4g_sample(const float *logits, int n_vocab, float temperature, float top_p,
                    uint64_t *rng_state, void *workspace, size_t workspace_bytes, void *stream)
{
    const int rc = sample_args_ok(logits, n_vocab, temperature, top_p, workspace, workspace_bytes);
    if (rc) return rc;
    unsigned u24 = 0;
    if (temperature > 0.f) {
        if (!rng_state || *rng_state == 0) return DS4G_EINVAL;
        u24 = (unsigned)(xorshift64s(rng_state) >> 40);
    }
    return sample_common(logits, n_vocab, temperature, top_p, 0.f, u24, workspace, workspace_bytes,
                         stream);
}

int32_t ds4g_sample_u(const float *logits, int n_vocab, float temperature, float top_p,
                      uint32_t u24, void *workspace, size_t workspace_bytes, void *stream)
{
    const int rc = sample_args_ok(logits, n_vocab, temperature, top_p, workspace, workspace_bytes);
    if (rc) return rc;
    if (u24 >= (1u << 24)) return DS4G_EINVAL;
    return sample_common(logits, n_vocab, temperature, top_p, 0.f, u24, workspace, workspace_bytes,
                         stream);
}

int32_t ds4g_sample_min_p(const float *logits, int n_vocab, float temperature, float top_p, float min_p,
                          uint64_t *rng_state, void *workspace, size_t workspace_bytes, void *stream)
{
    const int rc = sample_args_ok(logits, n_vocab, temperature, top_p, workspace, workspace_bytes);
    if (rc) return rc;
    if (!(min_p >= 0.f && min_p <= 1.f)) return DS4G_EINVAL;
    unsigned u24 = 0;
    if (temperature > 0.f) {
        if (!rng_state || *rng_state == 0) return DS4G_EINVAL;
        u24 = (unsigned)(xorshift64s(rng_state) >> 40);
    }
    return sample_common(logits, n_vocab, temperature, top_p, min_p, u24, workspace, workspace_bytes, stream);
}

int32_t ds4g_sample_u_min_p(const float *logits, int n_vocab, float temperature, float top_p, float min_p,
                            uint32_t u24, void *workspace, size_t workspace_bytes, void *stream)
{
    const int rc = sample_args_ok(logits, n_vocab, temperature, top_p, workspace, workspace_bytes);
    if (rc) return rc;
    if (!(min_p >= 0.f && min_p <= 1.f) || u24 >= (1u << 24)) return DS4G_EINVAL;
    return sample_common(logits, n_vocab, temperature, top_p, min_p, u24, workspace, workspace_bytes, stream);
}

static_assert(DS4G_SAMPLE_STATIC_MAX_VOCAB == kSampleStaticMaxVocab, "header and library agree");

int32_t ds4g_sample_static(const float *logits, int n_vocab, float temperature, float top_p,
                           uint64_t *rng_state, void *stream)
{
    if (!logits || n_vocab < 1 || temperature != temperature || top_p != top_p) return DS4G_EINVAL;
    if (n_vocab > DS4G_SAMPLE_STATIC_MAX_VOCAB) return DS4G_ESIZE;
    if (temperature > 0.f && (!rng_state || *rng_state == 0)) return DS4G_EINVAL;
    void *scratch = nullptr;
    if (sample_static_scratch(&scratch)) return DS4G_ECUDA;
    unsigned u24 = 0;
    if (temperature > 0.f) u24 = (unsigned)(xorshift64s(rng_state) >> 40);
    return sample_common(logits, n_vocab, temperature, top_p, 0.f, u24, scratch, kSampleStaticBytes, stream);
}

int32_t ds4g_decode_sample(ds4g_session *s, int32_t token, float temperature, float top_p, uint64_t *rng_state,
                           void *workspace, size_t workspace_bytes)
{
    if (!s) return DS4G_EINVAL;
    const int rc = sample_args_ok(s->b.logits, s->m->d.V, temperature, top_p, workspace, workspace_bytes);
    if (rc) return rc;
    if (temperature > 0.f && (!rng_state || *rng_state == 0)) return DS4G_EINVAL;
    const int drc = decode_common(s, token, true);
    if (drc) return drc;
    unsigned u24 = 0;
    if (temperature > 0.f) u24 = (unsigned)(xorshift64s(rng_state) >> 40);
    return sample_common(s->b.logits, s->m->d.V, temperature, top_p, 0.f, u24, workspace, workspace_bytes, s->st);
}

const char *ds4g_strerror(int code)
{
    switch (code) {
    case DS4G_OK: return "ok";
    case DS4G_EINVAL: return "invalid argument, shape or handle";
    case DS4G_ECONTEXT: return "tokens do not fit in the session context";
    case DS4G_ETOKEN: return "token id outside the vocabulary";
    case DS4G_ECUDA: return "CUDA call or kernel launch failed";
    case DS4G_ETIMEOUT: return "a bounded device-side wait gave up";
    case DS4G_ESIZE: return "buffer too small";
    case DS4G_ENONFINITE: return "a router score was not finite";
    default: return "unknown error";
    }
}

}  // extern "C"
