// Decode-step kernels: one token through one layer (page "ds4.c 学习笔记 --
// 端到端推理流程", 阶段四 4.2), and the lm_head (4.3).
//
// Batch-1 decode is bound by HBM: every kernel streams its weight rows once with
// 16-byte non-allocating loads and keeps the (small) activation vector in shared
// memory.  Design points:
//  - Grids are persistent (one CTA of 8 warps per SM, <= 128 registers) so that the
//    next kernel's CTA fits beside the current one.  Kernels are chained with
//    programmatic dependent launch: each kernel releases its successor right after
//    its prologue, and the successor, before waiting for its inputs, asks L2 to fetch
//    the weight rows of its first work item (weights do not depend on the token).
//    HBM therefore keeps streaming across kernel boundaries.
//  - Work items are dealt to warps CTA-interleaved (item i goes to SM i mod #SMs), so
//    even a small matrix spreads over every SM.
//  - A warp keeps a whole 8 KB row (or row pair) of loads in flight per round.
//  - Every reduction has a fixed order; results do not depend on timing.
#include "common.cuh"
#include "decode_common.cuh"
#include "kernels.h"

namespace ds4g {

static constexpr int kThreads = 256;

// ---- Q / KV down-projections: c = [W_qa; W_kva] * RMSNorm(x) ----------------------------
template <typename TW>
__global__ void __launch_bounds__(kThreads, 2) k_qkv_a(StepArgs a)
{
    extern __shared__ __align__(16) float smem[];
    float *xs = smem;
    float *red = smem + a.d.H;
    const int lane = threadIdx.x & 31, gw = gwarp(), gs = gwarps();
    const int H = a.d.H, nrows = a.d.RQ + a.d.RKV, nvec = H / VecOf<TW>::n;
    const TW *wqa = static_cast<const TW *>(a.w.wq_a), *wkva = static_cast<const TW *>(a.w.wkv_a);
    auto row = [&](int r) { return r < a.d.RQ ? wqa + (size_t)r * H : wkva + (size_t)(r - a.d.RQ) * H; };
    if (lane == 0 && gw < nrows) prefetch_l2(row(gw), H * sizeof(TW));
    const uint64_t pol = policy_evict_first();
    pdl_wait();
    float ss;
    if (a.token >= 0) {
        ss = load_f16_sumsq(a.tok_embd + (size_t)a.token * H, xs, H);
        __syncthreads();
        if (blockIdx.x == 0)
            for (int i = threadIdx.x * 4; i < H; i += blockDim.x * 4) {
                *reinterpret_cast<float4 *>(a.b.x + i) = *reinterpret_cast<float4 *>(xs + i);
                if (a.b.layer_x)   // recorded input of layer 0
                    *reinterpret_cast<float4 *>(a.b.layer_x + i) = *reinterpret_cast<float4 *>(xs + i);
            }
    } else {
        ss = load_f32_sumsq(a.b.x, xs, H);
    }
    finish_norm(ss, a.w.attn_norm, H, a.d.eps, xs, red);
    pdl_trigger();
    for (int r = gw; r < nrows; r += gs) {
        const TW *rows[1] = {row(r)};
        float acc[1] = {0.f};
        gemv_rows<TW, 1, 16>(rows, xs, nvec, acc, lane, pol);
        acc[0] = warp_sum(acc[0]);
        if (lane == 0) a.b.c[r] = acc[0];
    }
}

// ---- Q / K / V up-projections with RoPE and the KV-cache append ---------------------------
template <typename TW, typename TKV>
__global__ void __launch_bounds__(kThreads, 2) k_qkv_b(StepArgs a)
{
    extern __shared__ __align__(16) float smem[];
    float *xs = smem;  // [RQ + RKV]
    const int lane = threadIdx.x & 31, gw = gwarp(), gs = gwarps();
    const int HD = a.d.HD, nq = a.d.QD / 2, nk = HD / 2, RQ = a.d.RQ, RKV = a.d.RKV;
    const TW *wqb = static_cast<const TW *>(a.w.wq_b);
    const TW *wkb = static_cast<const TW *>(a.w.wk_b), *wvb = static_cast<const TW *>(a.w.wv_b);
    // pair u: rows (2p, 2p+1) of W_qb (u < nq), W_kb, or W_vb
    auto base_of = [&](int u, int &K, int &pr) -> const TW * {
        if (u < nq) { K = RQ; pr = u; return wqb; }
        K = RKV;
        if (u < nq + nk) { pr = u - nq; return wkb; }
        pr = u - nq - nk;
        return wvb;
    };
    if (lane == 0 && gw < nq + 2 * nk) {
        int K, pr;
        const TW *b = base_of(gw, K, pr);
        prefetch_l2(b + (size_t)(2 * pr) * K, 2 * K * sizeof(TW));
    }
    const uint64_t pol = policy_evict_first();
    pdl_wait();
    copy_f32(a.b.c, xs, RQ + RKV);
    __syncthreads();
    pdl_trigger();
    const float2 *rope = a.rope + (size_t)a.pos * (HD / 2);
    for (int u = gw; u < nq + 2 * nk; u += gs) {
        int K, pr;
        const TW *b = base_of(u, K, pr);
        const float *x = u < nq ? xs : xs + RQ;
        const TW *rows[2] = {b + (size_t)(2 * pr) * K, b + (size_t)(2 * pr + 1) * K};
        float acc[2] = {0.f, 0.f};
        gemv_rows<TW, 2, 4>(rows, x, K / VecOf<TW>::n, acc, lane, pol);
        float e = warp_sum(acc[0]), o = warp_sum(acc[1]);
        if (lane == 0) {
            if (u < nq + nk) {  // RoPE on the pair (2i, 2i+1) of a head
                const float2 cs = rope[pr % (HD / 2)];
                const float re = e * cs.x - o * cs.y, ro = e * cs.y + o * cs.x;
                e = re;
                o = ro;
            }
            if (u < nq) {
                a.b.q[2 * pr] = e;
                a.b.q[2 * pr + 1] = o;
            } else {
                TKV *dst = static_cast<TKV *>(u < nq + nk ? a.kc : a.vc) + (size_t)a.pos * HD;
                dst[2 * pr] = from_f32<TKV>(e);
                dst[2 * pr + 1] = from_f32<TKV>(o);
            }
        }
    }
}

// ---- sliding-window multi-query attention: one CTA per query head --------------------------
// The window's rows before `pos` were written by earlier steps, so they are staged
// (cp.async) before waiting for the up-projection kernel; only row `pos` and q after.
template <typename TKV>
__global__ void __launch_bounds__(128) k_attn(StepArgs a)
{
    extern __shared__ __align__(16) unsigned char sm[];
    const int HD = a.d.HD, W = a.d.W;
    TKV *Ks = reinterpret_cast<TKV *>(sm);
    TKV *Vs = Ks + (size_t)W * HD;
    float *qs = reinterpret_cast<float *>(Vs + (size_t)W * HD);
    float *ps = qs + HD;
    float *red = ps + W;
    const int h = blockIdx.x;
    const int lo = max(0, a.pos - W + 1), n = a.pos - lo + 1;
    const int vpr = HD * (int)sizeof(TKV) / 16;  // 16-byte vectors per row
    const uint4 *ksrc = reinterpret_cast<const uint4 *>(static_cast<const TKV *>(a.kc) + (size_t)lo * HD);
    const uint4 *vsrc = reinterpret_cast<const uint4 *>(static_cast<const TKV *>(a.vc) + (size_t)lo * HD);
    uint4 *kd = reinterpret_cast<uint4 *>(Ks), *vd = reinterpret_cast<uint4 *>(Vs);
    for (int i = threadIdx.x; i < (n - 1) * vpr; i += blockDim.x) {
        cp_async16(kd + i, ksrc + i);
        cp_async16(vd + i, vsrc + i);
    }
    pdl_wait();
    for (int i = (n - 1) * vpr + threadIdx.x; i < n * vpr; i += blockDim.x) {
        cp_async16(kd + i, ksrc + i);
        cp_async16(vd + i, vsrc + i);
    }
    const float scale = rsqrtf((float)HD);
    for (int d = threadIdx.x; d < HD; d += blockDim.x) qs[d] = a.b.q[(size_t)h * HD + d] * scale;
    cp_async_wait_all();
    __syncthreads();
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int j0 = warp * 4; j0 < n; j0 += nw * 4) {  // 4 keys per warp at a time
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        for (int d = lane; d < HD; d += 32) {
            const float qd = qs[d];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (j0 + u < n) s[u] = fmaf(qd, to_f32<TKV>(Ks[(size_t)(j0 + u) * HD + d]), s[u]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float t = warp_sum(s[u]);
            if (lane == 0 && j0 + u < n) ps[j0 + u] = t;
        }
    }
    __syncthreads();
    float m = -INFINITY;
    for (int j = threadIdx.x; j < n; j += blockDim.x) m = fmaxf(m, ps[j]);
    m = block_max(m, red);
    float sum = 0.f;
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
        const float e = __expf(ps[j] - m);
        ps[j] = e;
        sum += e;
    }
    sum = block_sum(sum, red);  // ends with a barrier: ps is complete
    const float inv = 1.f / sum;
    for (int d = threadIdx.x; d < HD; d += blockDim.x) {
        float acc = 0.f;
        for (int j = 0; j < n; ++j) acc = fmaf(ps[j], to_f32<TKV>(Vs[(size_t)j * HD + d]), acc);
        a.b.o[(size_t)h * HD + d] = acc * inv;
    }
}

// ---- attention output projection and residual: xm = x + W_o o ---------------------------
template <typename TW>
__global__ void __launch_bounds__(kThreads, 2) k_wo(StepArgs a)
{
    extern __shared__ __align__(16) float smem[];
    float *xs = smem;  // [QD]
    const int lane = threadIdx.x & 31, gw = gwarp(), gs = gwarps();
    const int QD = a.d.QD, nvec = QD / VecOf<TW>::n;
    const TW *wo = static_cast<const TW *>(a.w.wo);
    if (lane == 0 && gw < a.d.H) prefetch_l2(wo + (size_t)gw * QD, QD * sizeof(TW));
    const uint64_t pol = policy_evict_first();
    pdl_wait();
    copy_f32(a.b.o, xs, QD);
    __syncthreads();
    pdl_trigger();
    for (int r = gw; r < a.d.H; r += gs) {
        const TW *rows[1] = {wo + (size_t)r * QD};
        float acc[1] = {0.f};
        gemv_rows<TW, 1, 16>(rows, xs, nvec, acc, lane, pol);
        acc[0] = warp_sum(acc[0]);
        if (lane == 0) a.b.xm[r] = a.b.x[r] + acc[0];
    }
}

// ---- router: scores, top-k (ties to the lower id), softmax over the selected ----------------
// The last CTA to finish (grid ticket) takes the decision, so no second launch is needed.
template <typename TW>
__global__ void __launch_bounds__(kThreads, 2) k_router(StepArgs a)
{
    extern __shared__ __align__(16) float smem[];
    float *xs = smem;                          // [max(H, E)]
    float *red = smem + max(a.d.H, a.d.E);     // [32]
    __shared__ int s_last;
    const int lane = threadIdx.x & 31, gw = gwarp(), gs = gwarps();
    const int H = a.d.H, nvec = H / VecOf<TW>::n;
    const TW *wr = static_cast<const TW *>(a.w.w_router);
    if (lane == 0 && gw < a.d.E) prefetch_l2(wr + (size_t)gw * H, H * sizeof(TW));
    const uint64_t pol = policy_evict_first();
    pdl_wait();
    const float ss = load_f32_sumsq(a.b.xm, xs, H);
    finish_norm(ss, a.w.ffn_norm, H, a.d.eps, xs, red);
    pdl_trigger();
    if (blockIdx.x == 0)
        for (int i = threadIdx.x * 4; i < H; i += blockDim.x * 4)
            *reinterpret_cast<float4 *>(a.b.xn2 + i) = *reinterpret_cast<float4 *>(xs + i);
    for (int e = gw; e < a.d.E; e += gs) {
        const TW *rows[1] = {wr + (size_t)e * H};
        float acc[1] = {0.f};
        gemv_rows<TW, 1, 16>(rows, xs, nvec, acc, lane, pol);
        acc[0] = warp_sum(acc[0]);
        if (lane == 0) a.b.scores[e] = acc[0];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned t = atomicAdd(&a.b.counters[0], 1u);
        s_last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    float *sc = xs;  // reuse: [E]
    for (int e = threadIdx.x; e < a.d.E; e += blockDim.x) sc[e] = __ldcg(&a.b.scores[e]);
    __syncthreads();
    if (threadIdx.x < 32) {
        float sel[8];
        int ids[8];
        const bool finite = warp_topk(sc, a.d.E, a.d.K, sel, ids, lane);
        if (!finite && lane == 0) atomicCAS(a.b.status, 0, DS4G_ENONFINITE);
        if (lane == 0) {
            float sum = 0.f, wv[8];
            for (int k = 0; k < a.d.K; ++k) { wv[k] = expf(sel[k] - sel[0]); sum += wv[k]; }
            for (int k = 0; k < a.d.K; ++k) {
                a.b.ids[a.layer * a.d.K + k] = ids[k];
                a.b.wts[a.layer * a.d.K + k] = wv[k] / sum;
            }
            a.b.counters[0] = 0u;  // ready for the next layer
        }
    }
}

// ---- routed + shared experts, gate/up with SwiGLU: h_s = silu(Wg_e xn2) * (Wu_e xn2) -------
// Work item u < I is shared-expert row u (its weights are known before the router
// finishes and are prefetched); item I + s*I + i is row i of the s-th selected expert.
template <typename TW>
__global__ void __launch_bounds__(kThreads, 2) k_expert_gu(StepArgs a)
{
    extern __shared__ __align__(16) float smem[];
    float *xs = smem;  // [H]
    __shared__ int s_ids[8];
    const int lane = threadIdx.x & 31, gw = gwarp(), gs = gwarps();
    const int I = a.d.I, H = a.d.H, K = a.d.K, nvec = H / VecOf<TW>::n;
    const TW *wsg = static_cast<const TW *>(a.w.ws_gate), *wsu = static_cast<const TW *>(a.w.ws_up);
    if (lane == 0 && gw < I) {
        prefetch_l2(wsg + (size_t)gw * H, H * sizeof(TW));
        prefetch_l2(wsu + (size_t)gw * H, H * sizeof(TW));
    }
    const uint64_t pol = policy_evict_first();
    pdl_wait();
    copy_f32(a.b.xn2, xs, H);
    if (threadIdx.x < K) s_ids[threadIdx.x] = a.b.ids[a.layer * K + threadIdx.x];
    __syncthreads();
    pdl_trigger();
    for (int u = gw; u < (K + 1) * I; u += gs) {
        const TW *g, *up;
        int s, i;
        if (u < I) {
            s = K; i = u;
            g = wsg + (size_t)i * H;
            up = wsu + (size_t)i * H;
        } else {
            s = (u - I) / I; i = (u - I) - s * I;
            const size_t off = ((size_t)s_ids[s] * I + i) * H;
            g = static_cast<const TW *>(a.w.w_gate) + off;
            up = static_cast<const TW *>(a.w.w_up) + off;
        }
        const TW *rows[2] = {g, up};
        float acc[2] = {0.f, 0.f};
        gemv_rows<TW, 2, 8>(rows, xs, nvec, acc, lane, pol);
        const float gv = warp_sum(acc[0]), uv = warp_sum(acc[1]);
        if (lane == 0) a.b.h[(size_t)s * I + i] = gv / (1.f + expf(-gv)) * uv;
    }
}

// ---- expert down-projections, weighted combine and residual ------------------------------
// x = xm + sum_s w_s Wd_{e_s} h_s + Wd_shared h_shared for one output row pair per warp
// (shared expert first, then the selected experts in descending-score order).
template <typename TW>
__global__ void __launch_bounds__(kThreads, 2) k_expert_down(StepArgs a)
{
    extern __shared__ __align__(16) float smem[];
    float *hs = smem;  // [(K+1) * I]
    __shared__ int s_ids[8];
    __shared__ float s_w[9];
    const int lane = threadIdx.x & 31, gw = gwarp(), gs = gwarps();
    const int I = a.d.I, H = a.d.H, K = a.d.K;
    const TW *wsd = static_cast<const TW *>(a.w.ws_down);
    if (lane == 0 && 2 * gw < H) prefetch_l2(wsd + (size_t)(2 * gw) * I, 2 * I * sizeof(TW));
    const uint64_t pol = policy_evict_first();
    pdl_wait();
    copy_f32(a.b.h, hs, (K + 1) * I);
    if (threadIdx.x < K) {
        s_ids[threadIdx.x] = a.b.ids[a.layer * K + threadIdx.x];
        s_w[threadIdx.x] = a.b.wts[a.layer * K + threadIdx.x];
    }
    if (threadIdx.x == 0) s_w[K] = 1.f;
    __syncthreads();
    pdl_trigger();
    const int nvec = I / VecOf<TW>::n;
    for (int u = gw; u < H / 2; u += gs) {
        const int r0 = 2 * u;
        float tot[2] = {0.f, 0.f};
        for (int t = 0; t <= K; ++t) {
            const int s = t == 0 ? K : t - 1;
            const TW *base = s < K ? static_cast<const TW *>(a.w.w_down) + (size_t)s_ids[s] * H * I
                                   : wsd;
            const TW *rows[2] = {base + (size_t)r0 * I, base + (size_t)(r0 + 1) * I};
            float acc[2] = {0.f, 0.f};
            gemv_rows<TW, 2, 4>(rows, hs + (size_t)s * I, nvec, acc, lane, pol);
            tot[0] = fmaf(s_w[s], acc[0], tot[0]);
            tot[1] = fmaf(s_w[s], acc[1], tot[1]);
        }
        tot[0] = warp_sum(tot[0]);
        tot[1] = warp_sum(tot[1]);
        if (lane == 0) {
            a.b.x[r0] = a.b.xm[r0] + tot[0];
            a.b.x[r0 + 1] = a.b.xm[r0 + 1] + tot[1];
        }
    }
}

// ---- lm_head: logits = W_lm x (no final norm) ---------------------------------------------
template <typename TW>
__global__ void __launch_bounds__(kThreads, 2) k_lm_head(StepArgs a)
{
    extern __shared__ __align__(16) float smem[];
    float *xs = smem;  // [H]
    const int lane = threadIdx.x & 31, gw = gwarp(), gs = gwarps();
    const TW *lm = static_cast<const TW *>(a.lm_head);
    const int H = a.d.H, nvec = H / VecOf<TW>::n, V = a.d.V;
    if (lane == 0 && 2 * gw < V)
        prefetch_l2(lm + (size_t)(2 * gw) * H, (uint32_t)(min(2, V - 2 * gw) * H * sizeof(TW)));
    const uint64_t pol = policy_evict_first();
    pdl_wait();
    copy_f32(a.b.x, xs, H);
    __syncthreads();
    pdl_trigger();
    for (int u = gw; u < (V + 1) / 2; u += gs) {
        const int r0 = 2 * u, r1 = min(r0 + 1, V - 1);
        const TW *rows[2] = {lm + (size_t)r0 * H, lm + (size_t)r1 * H};
        float acc[2] = {0.f, 0.f};
        gemv_rows<TW, 2, 8>(rows, xs, nvec, acc, lane, pol);
        acc[0] = warp_sum(acc[0]);
        acc[1] = warp_sum(acc[1]);
        if (lane == 0) {
            a.b.logits[r0] = acc[0];
            if (r0 + 1 < V) a.b.logits[r0 + 1] = acc[1];
        }
    }
}

// ------------------------------------------------------------------ host side

static size_t attn_smem(const Dims &d)
{
    const size_t kvs = d.kvdt == DS4G_BF16 ? 2 : 4;
    return 2 * (size_t)d.W * d.HD * kvs + (size_t)(d.HD + d.W + 32) * 4;
}

template <typename TW, typename TKV>
static cudaError_t setup_t(const Dims &d, int big)
{
    cudaError_t e = cudaSuccess;
    auto set = [&](const void *f) {
        if (e == cudaSuccess) e = allow_max_dyn_smem(f, big);
    };
    set((const void *)k_qkv_a<TW>);
    set((const void *)k_qkv_b<TW, TKV>);
    set((const void *)k_attn<TKV>);
    set((const void *)k_wo<TW>);
    set((const void *)k_router<TW>);
    set((const void *)k_expert_gu<TW>);
    set((const void *)k_expert_down<TW>);
    set((const void *)k_lm_head<TW>);
    (void)d;
    return e;
}

cudaError_t decode_setup(const Dims &d, int max_smem)
{
    if (d.wdt == DS4G_BF16)
        return d.kvdt == DS4G_BF16 ? setup_t<bf16, bf16>(d, max_smem)
                                   : setup_t<bf16, float>(d, max_smem);
    return d.kvdt == DS4G_BF16 ? setup_t<float, bf16>(d, max_smem)
                               : setup_t<float, float>(d, max_smem);
}

// ev (optional): an event pair per kernel kind, recorded around each launch.
template <typename TW, typename TKV>
static cudaError_t layer_t(const StepArgs &a, cudaStream_t st, int nsm, cudaEvent_t (*ev)[2])
{
    const Dims &d = a.d;
    const dim3 g(nsm), b(kThreads);
    cudaError_t e;
    auto mark = [&](int k, int w) { if (ev) cudaEventRecord(ev[k][w], st); };
    StepArgs first = a;
    mark(DS4G_K_QKV_A, 0);
    if ((e = launch_pdl(k_qkv_a<TW>, g, b, (d.H + 32) * 4, st, first))) return e;
    mark(DS4G_K_QKV_A, 1);
    StepArgs rest = a;
    rest.token = -1;
    mark(DS4G_K_QKV_B, 0);
    if ((e = launch_pdl(k_qkv_b<TW, TKV>, g, b, (d.RQ + d.RKV) * 4, st, rest))) return e;
    mark(DS4G_K_QKV_B, 1);
    mark(DS4G_K_ATTN, 0);
    if ((e = launch_pdl(k_attn<TKV>, dim3(d.NH), dim3(128), attn_smem(d), st, rest))) return e;
    mark(DS4G_K_ATTN, 1);
    mark(DS4G_K_WO, 0);
    if ((e = launch_pdl(k_wo<TW>, g, b, d.QD * 4, st, rest))) return e;
    mark(DS4G_K_WO, 1);
    const int rsm = ((d.H > d.E ? d.H : d.E) + 32) * 4;
    mark(DS4G_K_ROUTER, 0);
    if ((e = launch_pdl(k_router<TW>, g, b, rsm, st, rest))) return e;
    mark(DS4G_K_ROUTER, 1);
    mark(DS4G_K_EXPERT_GU, 0);
    if ((e = launch_pdl(k_expert_gu<TW>, g, b, d.H * 4, st, rest))) return e;
    mark(DS4G_K_EXPERT_GU, 1);
    mark(DS4G_K_EXPERT_DOWN, 0);
    if ((e = launch_pdl(k_expert_down<TW>, g, b, (d.K + 1) * d.I * 4, st, rest))) return e;
    mark(DS4G_K_EXPERT_DOWN, 1);
    return cudaSuccess;
}

cudaError_t decode_layer(const StepArgs &a, cudaStream_t st, int nsm, cudaEvent_t (*ev)[2])
{
    const Dims &d = a.d;
    if (d.wdt == DS4G_BF16)
        return d.kvdt == DS4G_BF16 ? layer_t<bf16, bf16>(a, st, nsm, ev)
                                   : layer_t<bf16, float>(a, st, nsm, ev);
    return d.kvdt == DS4G_BF16 ? layer_t<float, bf16>(a, st, nsm, ev)
                               : layer_t<float, float>(a, st, nsm, ev);
}

cudaError_t decode_lm_head(const StepArgs &a, cudaStream_t st, int nsm)
{
    const Dims &d = a.d;
    if (d.wdt == DS4G_BF16)
        return launch_pdl(k_lm_head<bf16>, dim3(nsm), dim3(kThreads), d.H * 4, st, a);
    return launch_pdl(k_lm_head<float>, dim3(nsm), dim3(kThreads), d.H * 4, st, a);
}

}  // namespace ds4g
