// Decode-step kernels: one token through one layer (page "ds4.c 学习笔记 --
// 端到端推理流程", 阶段四 4.2), and the lm_head (4.3).
//
// Batch-1 decode is bound by HBM: every kernel streams its weight rows once
// with 16-byte non-allocating loads and keeps the (small) activation vector in
// shared memory.  Grids are persistent (one CTA per SM, 16 warps); kernels are
// chained with programmatic dependent launch so that a kernel's CTAs are
// resident and its first weight loads can be issued while the previous kernel
// drains.  Every reduction has a fixed order, so results do not depend on
// timing.
#include "common.cuh"
#include "kernels.h"

namespace ds4g {

static constexpr int kThreads = 512;
static constexpr int kWarps = kThreads / 32;

// RMSNorm of a length-H vector into shared memory: xs = v * rsqrt(mean(v^2) + eps) * g.
// `src` is f32 (the residual) or, for the first layer, an f16 embedding row.
template <typename TSrc>
__device__ __forceinline__ void norm_into_smem(const TSrc *src, const float *g, int H, float eps,
                                               float *xs, float *red, float *raw_out)
{
    float ss = 0.f;
    for (int i = threadIdx.x; i < H; i += blockDim.x) {
        float v;
        if constexpr (sizeof(TSrc) == 2)
            v = __half2float(reinterpret_cast<const __half *>(src)[i]);
        else
            v = src[i];
        xs[i] = v;
        ss = fmaf(v, v, ss);
        if (raw_out) raw_out[i] = v;
    }
    ss = block_sum(ss, red);
    const float inv = rsqrtf(ss / (float)H + eps);
    for (int i = threadIdx.x; i < H; i += blockDim.x) xs[i] = xs[i] * inv * g[i];
    __syncthreads();
}

// ---- Q / KV down-projections: c = [W_qa; W_kva] * RMSNorm(x) ----------------------------
template <typename TW>
__global__ void __launch_bounds__(kThreads) k_qkv_a(StepArgs a)
{
    extern __shared__ __align__(16) float smem[];
    float *xs = smem;
    float *red = smem + a.d.H;
    const uint64_t pol = policy_evict_first();
    pdl_wait();
    if (a.token >= 0) {
        const uint16_t *row = a.tok_embd + (size_t)a.token * a.d.H;
        norm_into_smem<uint16_t>(row, a.w.attn_norm, a.d.H, a.d.eps, xs, red,
                                 blockIdx.x == 0 ? a.b.x : nullptr);
    } else {
        norm_into_smem<float>(a.b.x, a.w.attn_norm, a.d.H, a.d.eps, xs, red, nullptr);
    }
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5), gs = gridDim.x * kWarps;
    const int nrows = a.d.RQ + a.d.RKV, nvec = a.d.H / VecOf<TW>::n;
    const TW *wqa = static_cast<const TW *>(a.w.wq_a), *wkva = static_cast<const TW *>(a.w.wkv_a);
    for (int u = gw; u < nrows / 2; u += gs) {
        const int r0 = 2 * u;
        const TW *rows[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int r = r0 + j;
            rows[j] = r < a.d.RQ ? wqa + (size_t)r * a.d.H : wkva + (size_t)(r - a.d.RQ) * a.d.H;
        }
        float acc[2] = {0.f, 0.f};
        gemv_rows<TW, 2, 4>(rows, xs, nvec, acc, lane, pol);
        acc[0] = warp_sum(acc[0]);
        acc[1] = warp_sum(acc[1]);
        if (lane == 0) {
            a.b.c[r0] = acc[0];
            a.b.c[r0 + 1] = acc[1];
        }
    }
}

// ---- Q / K / V up-projections with RoPE and the KV-cache append ---------------------------
template <typename TW, typename TKV>
__global__ void __launch_bounds__(kThreads) k_qkv_b(StepArgs a)
{
    extern __shared__ __align__(16) float smem[];
    float *xs = smem;  // [RQ + RKV]
    const uint64_t pol = policy_evict_first();
    pdl_wait();
    const int nc = a.d.RQ + a.d.RKV;
    for (int i = threadIdx.x; i < nc; i += blockDim.x) xs[i] = a.b.c[i];
    __syncthreads();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5), gs = gridDim.x * kWarps;
    const int HD = a.d.HD, nq = a.d.QD / 2, nk = HD / 2;
    const float2 *rope = a.rope + (size_t)a.pos * (HD / 2);
    for (int u = gw; u < nq + 2 * nk; u += gs) {
        const TW *base;
        const float *x;
        int K, pr;  // pair index within its matrix
        if (u < nq) {
            base = static_cast<const TW *>(a.w.wq_b); x = xs; K = a.d.RQ; pr = u;
        } else if (u < nq + nk) {
            base = static_cast<const TW *>(a.w.wk_b); x = xs + a.d.RQ; K = a.d.RKV; pr = u - nq;
        } else {
            base = static_cast<const TW *>(a.w.wv_b); x = xs + a.d.RQ; K = a.d.RKV; pr = u - nq - nk;
        }
        const TW *rows[2] = {base + (size_t)(2 * pr) * K, base + (size_t)(2 * pr + 1) * K};
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
    pdl_wait();
    const int lo = max(0, a.pos - W + 1), n = a.pos - lo + 1;
    // stage the window's K and V rows (contiguous in the cache) with 16-byte copies
    const int nv = n * HD * (int)sizeof(TKV) / 16;
    const uint4 *ksrc = reinterpret_cast<const uint4 *>(static_cast<const TKV *>(a.kc) + (size_t)lo * HD);
    const uint4 *vsrc = reinterpret_cast<const uint4 *>(static_cast<const TKV *>(a.vc) + (size_t)lo * HD);
    for (int i = threadIdx.x; i < nv; i += blockDim.x) {
        reinterpret_cast<uint4 *>(Ks)[i] = ksrc[i];
        reinterpret_cast<uint4 *>(Vs)[i] = vsrc[i];
    }
    const float scale = rsqrtf((float)HD);
    for (int d = threadIdx.x; d < HD; d += blockDim.x) qs[d] = a.b.q[(size_t)h * HD + d] * scale;
    __syncthreads();
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int j = warp; j < n; j += nw) {
        float s = 0.f;
        for (int d = lane; d < HD; d += 32) s = fmaf(qs[d], to_f32<TKV>(Ks[(size_t)j * HD + d]), s);
        s = warp_sum(s);
        if (lane == 0) ps[j] = s;
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
__global__ void __launch_bounds__(kThreads) k_wo(StepArgs a)
{
    extern __shared__ __align__(16) float smem[];
    float *xs = smem;  // [QD]
    const uint64_t pol = policy_evict_first();
    pdl_wait();
    for (int i = threadIdx.x; i < a.d.QD; i += blockDim.x) xs[i] = a.b.o[i];
    __syncthreads();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5), gs = gridDim.x * kWarps;
    const TW *wo = static_cast<const TW *>(a.w.wo);
    const int nvec = a.d.QD / VecOf<TW>::n;
    for (int u = gw; u < a.d.H / 2; u += gs) {
        const int r0 = 2 * u;
        const TW *rows[2] = {wo + (size_t)r0 * a.d.QD, wo + (size_t)(r0 + 1) * a.d.QD};
        float acc[2] = {0.f, 0.f};
        gemv_rows<TW, 2, 4>(rows, xs, nvec, acc, lane, pol);
        acc[0] = warp_sum(acc[0]);
        acc[1] = warp_sum(acc[1]);
        if (lane == 0) {
            a.b.xm[r0] = a.b.x[r0] + acc[0];
            a.b.xm[r0 + 1] = a.b.x[r0 + 1] + acc[1];
        }
    }
}

// ---- router: scores, top-k (ties to the lower id), softmax over the selected ----------------
// The last CTA to finish (grid ticket) takes the decision, so no second launch is needed.
template <typename TW>
__global__ void __launch_bounds__(kThreads) k_router(StepArgs a)
{
    extern __shared__ __align__(16) float smem[];
    float *xs = smem;                          // [max(H, E)]
    float *red = smem + max(a.d.H, a.d.E);     // [32]
    __shared__ int s_last;
    const uint64_t pol = policy_evict_first();
    pdl_wait();
    norm_into_smem<float>(a.b.xm, a.w.ffn_norm, a.d.H, a.d.eps, xs, red, nullptr);
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < a.d.H; i += blockDim.x) a.b.xn2[i] = xs[i];
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5), gs = gridDim.x * kWarps;
    const TW *wr = static_cast<const TW *>(a.w.w_router);
    const int nvec = a.d.H / VecOf<TW>::n;
    for (int e = gw; e < a.d.E; e += gs) {
        const TW *rows[1] = {wr + (size_t)e * a.d.H};
        float acc[1] = {0.f};
        gemv_rows<TW, 1, 8>(rows, xs, nvec, acc, lane, pol);
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
    // top-k by repeated warp arg-max over the scores copied to shared memory
    float *sc = xs;  // reuse: [E]
    for (int e = threadIdx.x; e < a.d.E; e += blockDim.x) sc[e] = __ldcg(&a.b.scores[e]);
    __syncthreads();
    if (threadIdx.x < 32) {
        float sel[8];
        int ids[8];
        for (int k = 0; k < a.d.K; ++k) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            for (int e = lane; e < a.d.E; e += 32) {
                const float v = sc[e];
                if (v > bv || (v == bv && e < bi)) { bv = v; bi = e; }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            sel[k] = bv;
            ids[k] = bi;
            __syncwarp();
            if (lane == 0) sc[bi] = -INFINITY;
            __syncwarp();
        }
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
template <typename TW>
__global__ void __launch_bounds__(kThreads) k_expert_gu(StepArgs a)
{
    extern __shared__ __align__(16) float smem[];
    float *xs = smem;  // [H]
    __shared__ int s_ids[9];
    const uint64_t pol = policy_evict_first();
    pdl_wait();
    for (int i = threadIdx.x; i < a.d.H; i += blockDim.x) xs[i] = a.b.xn2[i];
    if (threadIdx.x < a.d.K) s_ids[threadIdx.x] = a.b.ids[a.layer * a.d.K + threadIdx.x];
    __syncthreads();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5), gs = gridDim.x * kWarps;
    const int I = a.d.I, H = a.d.H, K = a.d.K, nvec = H / VecOf<TW>::n;
    for (int u = gw; u < (K + 1) * I; u += gs) {
        const int s = u / I, i = u - s * I;
        const TW *g, *up;
        if (s < K) {
            const size_t off = ((size_t)s_ids[s] * I + i) * H;
            g = static_cast<const TW *>(a.w.w_gate) + off;
            up = static_cast<const TW *>(a.w.w_up) + off;
        } else {
            g = static_cast<const TW *>(a.w.ws_gate) + (size_t)i * H;
            up = static_cast<const TW *>(a.w.ws_up) + (size_t)i * H;
        }
        const TW *rows[2] = {g, up};
        float acc[2] = {0.f, 0.f};
        gemv_rows<TW, 2, 4>(rows, xs, nvec, acc, lane, pol);
        const float gv = warp_sum(acc[0]), uv = warp_sum(acc[1]);
        if (lane == 0) a.b.h[u] = gv / (1.f + expf(-gv)) * uv;
    }
}

// ---- expert down-projections, weighted combine and residual ------------------------------
// x = xm + sum_s w_s Wd_{e_s} h_s + Wd_shared h_shared, one output row pair per warp.
template <typename TW>
__global__ void __launch_bounds__(kThreads) k_expert_down(StepArgs a)
{
    extern __shared__ __align__(16) float smem[];
    float *hs = smem;  // [(K+1) * I]
    __shared__ int s_ids[8];
    __shared__ float s_w[9];
    const uint64_t pol = policy_evict_first();
    pdl_wait();
    const int I = a.d.I, H = a.d.H, K = a.d.K;
    for (int i = threadIdx.x; i < (K + 1) * I; i += blockDim.x) hs[i] = a.b.h[i];
    if (threadIdx.x < K) {
        s_ids[threadIdx.x] = a.b.ids[a.layer * K + threadIdx.x];
        s_w[threadIdx.x] = a.b.wts[a.layer * K + threadIdx.x];
    }
    if (threadIdx.x == 0) s_w[K] = 1.f;
    __syncthreads();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5), gs = gridDim.x * kWarps;
    const int nvec = I / VecOf<TW>::n;
    for (int u = gw; u < H / 2; u += gs) {
        const int r0 = 2 * u;
        float tot[2] = {0.f, 0.f};
        for (int s = 0; s <= K; ++s) {
            const TW *base = s < K ? static_cast<const TW *>(a.w.w_down) + (size_t)s_ids[s] * H * I
                                   : static_cast<const TW *>(a.w.ws_down);
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
__global__ void __launch_bounds__(kThreads) k_lm_head(StepArgs a)
{
    extern __shared__ __align__(16) float smem[];
    float *xs = smem;  // [H]
    const uint64_t pol = policy_evict_first();
    pdl_wait();
    for (int i = threadIdx.x; i < a.d.H; i += blockDim.x) {
        const float v = a.b.x[i];
        xs[i] = v;
        if (blockIdx.x == 0) a.b.hidden[i] = v;
    }
    __syncthreads();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5), gs = gridDim.x * kWarps;
    const TW *lm = static_cast<const TW *>(a.lm_head);
    const int nvec = a.d.H / VecOf<TW>::n, V = a.d.V;
    for (int u = gw; u < (V + 1) / 2; u += gs) {
        const int r0 = 2 * u, r1 = min(r0 + 1, V - 1);
        const TW *rows[2] = {lm + (size_t)r0 * a.d.H, lm + (size_t)r1 * a.d.H};
        float acc[2] = {0.f, 0.f};
        gemv_rows<TW, 2, 4>(rows, xs, nvec, acc, lane, pol);
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
    const int rblocks = (d.E + kWarps - 1) / kWarps;
    const int rsm = ((d.H > d.E ? d.H : d.E) + 32) * 4;
    mark(DS4G_K_ROUTER, 0);
    if ((e = launch_pdl(k_router<TW>, dim3(rblocks < nsm ? rblocks : nsm), b, rsm, st, rest)))
        return e;
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
