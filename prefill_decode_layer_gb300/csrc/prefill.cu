// Layer-major prefill (page "ds4.c 学习笔记 -- 端到端推理流程", 阶段三
// prefill_layer_major_cpu): layer l runs over every token of the chunk before
// layer l+1, so each layer's weights are streamed once per chunk.
//
// Per layer: RMSNorm -> [W_qa; W_kva] GEMM -> W_qb GEMM with RoPE -> [W_kb; W_vb]
// GEMM with RoPE and the KV-cache append -> windowed causal MQA -> W_o GEMM with
// the residual -> RMSNorm -> router GEMM -> per-token top-k -> tokens grouped per
// expert (stable counting sort) -> grouped gate/up GEMMs with SwiGLU -> shared
// expert -> grouped down GEMMs scattered per (token, slot) -> shared down GEMM
// whose epilogue adds the weighted routed outputs in slot order and the residual.
//
// Every output element is accumulated in a fixed order that does not depend on
// how many tokens share the chunk, so a token's results are the same whether it
// is prefilled alone, in a suffix after a truncation, or inside a long prompt.
//
// The GEMMs here are SIMT tiles with f32 activations and f32 accumulation.
#include "common.cuh"
#include "gemm.cuh"
#include "kernels.h"
#include "prefill_problems.cuh"
#include "prefill_tc.h"

namespace ds4g {

// ------------------------------------------------------------------ small kernels

__global__ void k_embed_rows(const uint16_t *table, const int *tok, float *X, int H)
{
    pdl_wait();      // inputs of the previous kernel (programmatic launch)
    pdl_trigger();
    const int t = blockIdx.x;
    const __half *row = reinterpret_cast<const __half *>(table) + (size_t)tok[t] * H;
    for (int i = threadIdx.x; i < H; i += blockDim.x) X[(size_t)t * H + i] = __half2float(row[i]);
}

// out = RMSNorm(X) in the activation type; out32 (optional) keeps an f32 copy for
// the router, whose top-k decisions need more than bf16 input precision.
template <typename TA>
__global__ void __launch_bounds__(256) k_rmsnorm_rows(const float *X, const float *g, TA *out,
                                                      float *out32, int H, float eps)
{
    __shared__ float red[32];
    const int t = blockIdx.x;
    const float *x = X + (size_t)t * H;
    float ss = 0.f;
    for (int i = threadIdx.x; i < H; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
    ss = block_sum(ss, red);
    const float inv = rsqrtf(ss / (float)H + eps);
    for (int i = threadIdx.x; i < H; i += blockDim.x) {
        const float y = x[i] * inv * g[i];
        out[(size_t)t * H + i] = from_f32<TA>(y);
        if (out32) out32[(size_t)t * H + i] = y;
    }
}

// Router decision per token: top-k of the scores (ties to the lower id), softmax
// over the selected scores.  One warp per token.  The scores may come as two
// partial sums (of the reduction's two parts, `part` elements apart; E <= 256),
// added in part order (nparts 2; otherwise 1).
__global__ void k_router_topk(const float *S, int nparts, size_t part, int *ids, float *wts, int n, int E, int K,
                              int *status)
{
    pdl_wait();      // inputs of the previous kernel (programmatic launch)
    pdl_trigger();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= n) return;
    float sel[8];
    int sid[8];
    bool finite;
    if (nparts == 2) {   // both parts' loads in flight before the adds
        const float *s0 = S + (size_t)warp * E, *s1 = s0 + part;
        float x[8], y[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = lane + 32 * u;
            x[u] = e < E ? s0[e] : 0.f;
            y[u] = e < E ? s1[e] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] += y[u];
        finite = warp_topk_r256(x, E, K, sel, sid, lane);
    } else {
        finite = warp_topk(S + (size_t)warp * E, E, K, sel, sid, lane);
    }
    if (!finite && lane == 0) atomicCAS(status, 0, DS4G_ENONFINITE);
    if (lane == 0) {
        float sum = 0.f, w[8];
        for (int k = 0; k < K; ++k) { w[k] = expf(sel[k] - sel[0]); sum += w[k]; }
        for (int k = 0; k < K; ++k) {
            ids[(size_t)warp * K + k] = sid[k];
            wts[(size_t)warp * K + k] = w[k] / sum;
        }
    }
}

// Stable grouping of the (token, slot) entries by expert: a counting sort in three
// passes over segments of kSortSeg entries.  Entry i = token * K + slot; an
// expert's rows come out in increasing i, so the grouped order depends only on
// the ids.  Pass 1: per-segment histograms (shared-memory atomics).
__global__ void __launch_bounds__(256) k_group_hist(const int *ids, int nent, int E, int *segcnt)
{
    pdl_wait();      // inputs of the previous kernel (programmatic launch)
    pdl_trigger();
    extern __shared__ int hist[];
    const int seg = blockIdx.x, i0 = seg * kSortSeg, i1 = min(nent, i0 + kSortSeg);
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
        const int id = ids[i];
        if ((unsigned)id < (unsigned)E) atomicAdd(&hist[id], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) segcnt[(size_t)seg * E + e] = hist[e];
}

// Exclusive scan over the block's threads (blockDim.x a multiple of 32, <= 1024).
__device__ int block_exclusive_scan(int v, int *tmp, int &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? tmp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nw) tmp[lane] = w;   // inclusive warp totals
    }
    __syncthreads();
    total = tmp[nw - 1];
    const int r = x - v + (warp ? tmp[warp - 1] : 0);
    __syncthreads();   // tmp may be reused
    return r;
}

// Pass 2 (one CTA): each expert's count and its segments' exclusive prefixes
// (segcnt is rewritten in place), the expert offsets, and the (expert, first row)
// tile list, tiles of bm rows that never cross an expert boundary.  Thread t owns
// the experts [t * per, (t + 1) * per).
__global__ void __launch_bounds__(1024) k_group_offsets(int *segcnt, int nseg, int E, int bm, int *cnt, int *off,
                                                        int *tiles)
{
    pdl_wait();      // inputs of the previous kernel (programmatic launch)
    pdl_trigger();
    __shared__ int tmp[32];
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = min(E, (int)threadIdx.x * per), e1 = min(E, e0 + per);
    int rows = 0, ntile = 0;
    for (int e = e0; e < e1; ++e) {
        int run = 0;
        int s = 0;
        for (; s + 8 <= nseg; s += 8) {   // eight independent loads in flight
            int c[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) c[j] = segcnt[(size_t)(s + j) * E + e];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                segcnt[(size_t)(s + j) * E + e] = run;
                run += c[j];
            }
        }
        for (; s < nseg; ++s) {
            const int c = segcnt[(size_t)s * E + e];
            segcnt[(size_t)s * E + e] = run;
            run += c;
        }
        cnt[e] = run;
        rows += run;
        ntile += (run + bm - 1) / bm;
    }
    int nrows, ntiles;
    int o = block_exclusive_scan(rows, tmp, nrows);
    int t = block_exclusive_scan(ntile, tmp, ntiles);
    for (int e = e0; e < e1; ++e) {
        const int c = cnt[e];
        off[e] = o;
        for (int r = 0; r < c; r += bm, ++t) {
            tiles[1 + 2 * t] = e;
            tiles[2 + 2 * t] = o + r;
        }
        o += c;
    }
    if (threadIdx.x == 0) {
        off[E] = nrows;
        tiles[0] = ntiles;
    }
}

// Pass 3: one warp per segment places its entries in index order.  Lanes holding
// the same expert find one another with a match, rank by lane, and the group's
// last lane advances the expert's running base.
__global__ void __launch_bounds__(32) k_group_place(const int *ids, int nent, int E, const int *segcnt,
                                                    const int *off, int *rows)
{
    pdl_wait();      // inputs of the previous kernel (programmatic launch)
    pdl_trigger();
    extern __shared__ int base[];
    const int seg = blockIdx.x, lane = threadIdx.x;
    const int i0 = seg * kSortSeg, i1 = min(nent, i0 + kSortSeg);
    for (int e = lane; e < E; e += 32) base[e] = off[e] + segcnt[(size_t)seg * E + e];
    __syncwarp();
    for (int c = i0; c < i1; c += 32) {
        const int i = c + lane;
        int id = i < i1 ? ids[i] : -1;
        const bool ok = (unsigned)id < (unsigned)E;
        if (!ok) id = -1 - lane;   // matches no other lane
        const unsigned peers = __match_any_sync(0xffffffffu, id);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        int b = 0;
        if (ok) b = base[id];
        __syncwarp();
        if (ok) {
            rows[b + rank] = i;
            if (rank == __popc(peers) - 1) base[id] = b + rank + 1;
        }
        __syncwarp();
    }
}

cudaError_t group_by_expert(const PrefillBufs &pb, int nent, int E, int bm, cudaStream_t st)
{
    const int nseg = (nent + kSortSeg - 1) / kSortSeg;
    if (nseg == 0) {
        cudaError_t e = cudaMemsetAsync(pb.tiles, 0, sizeof(int), st);
        if (e) return e;
        return cudaMemsetAsync(pb.off, 0, (size_t)(E + 1) * sizeof(int), st);
    }
    const size_t sh = (size_t)E * sizeof(int);
    cudaError_t e = launch_pdl(k_group_hist, dim3(nseg), dim3(256), sh, st, (const int *)pb.ids, nent, E, pb.segcnt);
    const int thr = E >= 1024 ? 1024 : ((E + 31) / 32) * 32;
    if (!e)
        e = launch_pdl(k_group_offsets, dim3(1), dim3(thr), 0, st, pb.segcnt, nseg, E, bm, pb.cnt, pb.off, pb.tiles);
    if (!e)
        e = launch_pdl(k_group_place, dim3(nseg), dim3(32), sh, st, (const int *)pb.ids, nent, E,
                       (const int *)pb.segcnt, (const int *)pb.off, pb.rows);
    return e;
}

// Windowed causal multi-query attention for a chunk: CTA (token t, group of heads).
// The window's K/V rows are staged once in shared memory for all heads of the group.
// HILO: the output is written as BF16 hi/lo pairs (O and Olo) for the tensor-core
// W_o GEMM instead of in the activation type.
template <typename TA, typename TKV, bool HILO = false>
__global__ void __launch_bounds__(256) k_attn_prefill(const TA *Q, void *Ov, bf16 *Olo, const TKV *kc,
                                                      const TKV *vc, int p0, Dims d, int hg)
{
    extern __shared__ __align__(16) unsigned char sm[];
    const int HD = d.HD, W = d.W;
    TKV *Ks = reinterpret_cast<TKV *>(sm);
    TKV *Vs = Ks + (size_t)W * HD;
    float *qs = reinterpret_cast<float *>(Vs + (size_t)W * HD);  // [8 warps][HD]
    float *ps = qs + 8 * HD;                                     // [8 warps][W]
    const int t = blockIdx.x, pos = p0 + t;
    const int lo = max(0, pos - W + 1), n = pos - lo + 1;
    const int nv = n * HD * (int)sizeof(TKV) / 16;
    const uint4 *ks = reinterpret_cast<const uint4 *>(kc + (size_t)lo * HD);
    const uint4 *vs = reinterpret_cast<const uint4 *>(vc + (size_t)lo * HD);
    for (int i = threadIdx.x; i < nv; i += blockDim.x) {
        reinterpret_cast<uint4 *>(Ks)[i] = ks[i];
        reinterpret_cast<uint4 *>(Vs)[i] = vs[i];
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float scale = rsqrtf((float)HD);
    float *q = qs + warp * HD, *p = ps + warp * W;
    for (int hh = warp; hh < hg; hh += 8) {
        const int h = blockIdx.y * hg + hh;
        if (h >= d.NH) break;
        const TA *qrow = Q + (size_t)t * d.QD + (size_t)h * HD;
        for (int i = lane; i < HD; i += 32) q[i] = to_f32<TA>(qrow[i]) * scale;
        __syncwarp();
        // scores: lanes split the head dimension (conflict-free rows), 4 keys at a time
        float m = -INFINITY;
        for (int j0 = 0; j0 < n; j0 += 4) {
            float s[4] = {0.f, 0.f, 0.f, 0.f};
            for (int i = lane; i < HD; i += 32) {
                const float qi = q[i];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (j0 + u < n) s[u] = fmaf(qi, to_f32<TKV>(Ks[(size_t)(j0 + u) * HD + i]), s[u]);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                s[u] = warp_sum(s[u]);
                if (j0 + u < n) {
                    m = fmaxf(m, s[u]);
                    if (lane == 0) p[j0 + u] = s[u];
                }
            }
        }
        __syncwarp();
        float sum = 0.f;
        for (int j = lane; j < n; j += 32) {
            const float e = __expf(p[j] - m);
            p[j] = e;
            sum += e;
        }
        sum = warp_sum(sum);
        __syncwarp();
        const float inv = 1.f / sum;
        for (int i = lane; i < HD; i += 32) {
            float acc = 0.f;
            for (int j = 0; j < n; ++j) acc = fmaf(p[j], to_f32<TKV>(Vs[(size_t)j * HD + i]), acc);
            const size_t oi = (size_t)t * d.QD + (size_t)h * HD + i;
            if constexpr (HILO) {
                const float ov = acc * inv;
                const bf16 hv = __float2bfloat16_rn(ov);
                static_cast<bf16 *>(Ov)[oi] = hv;
                Olo[oi] = __float2bfloat16_rn(ov - __bfloat162float(hv));
            } else {
                static_cast<TA *>(Ov)[oi] = from_f32<TA>(acc * inv);
            }
        }
        __syncwarp();
    }
}

// ------------------------------------------------------------------ host side

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

void prefill_carve(const Dims &d, int P, char *base, PrefillBufs &pb)
{
    const size_t ta = 4;
    const size_t PK = (size_t)P * d.K;
    size_t o = 0;   // offsets as integers: prefill_bytes walks from a null base
    auto take = [&](size_t n) {
        const size_t r = o;
        o += align256(n);
        return reinterpret_cast<void *>(reinterpret_cast<uintptr_t>(base) + r);
    };
    pb.P = P;
    pb.tok = (int *)take((size_t)P * 4);
    pb.X = (float *)take((size_t)P * d.H * 4);
    pb.XN = take((size_t)P * d.H * ta);
    pb.XN32 = (float *)take((size_t)P * d.H * 4);
    pb.C = take((size_t)P * (d.RQ + d.RKV) * ta);
    pb.Q = take((size_t)P * d.QD * ta);
    pb.O = take((size_t)P * d.QD * ta);
    pb.S = (float *)take((size_t)kRouterParts * P * d.E * 4);
    pb.ids = (int *)take(PK * 4);
    pb.wts = (float *)take(PK * 4);
    pb.cnt = (int *)take((size_t)d.E * 4);
    pb.off = (int *)take((size_t)(d.E + 1) * 4);
    pb.rows = (int *)take(PK * 4);
    pb.segcnt = (int *)take(sort_segments(PK) * d.E * 4);
    pb.tiles = (int *)take((PK / 16 + d.E + 2) * 2 * 4);
    pb.HG = take(PK * d.I * ta);
    pb.HS = take((size_t)P * d.I * ta);
    pb.YS = (float *)take(PK * d.H * 4);
    pb.end = reinterpret_cast<char *>(reinterpret_cast<uintptr_t>(base) + o);
}

// The bytes prefill_carve lays out (the same walk from address 0).
size_t prefill_bytes(const Dims &d, int P)
{
    PrefillBufs pb{};
    prefill_carve(d, P, nullptr, pb);
    return (size_t)reinterpret_cast<uintptr_t>(pb.end);
}

static size_t attn_prefill_smem(const Dims &d)
{
    const size_t kvs = d.kvdt == DS4G_BF16 ? 2 : 4;
    return 2 * (size_t)d.W * d.HD * kvs + 8 * (size_t)(d.HD + d.W) * 4;
}

cudaError_t prefill_setup(const Dims &d, int max_smem)
{
    cudaError_t e = d.kvdt == DS4G_BF16
                        ? allow_max_dyn_smem((const void *)k_attn_prefill<float, bf16>, max_smem)
                        : allow_max_dyn_smem((const void *)k_attn_prefill<float, float>, max_smem);
    if (e) return e;
    return d.kvdt == DS4G_BF16 ? allow_max_dyn_smem((const void *)k_attn_prefill<float, bf16, true>, max_smem)
                               : allow_max_dyn_smem((const void *)k_attn_prefill<float, float, true>, max_smem);
}

template <typename TKV>
cudaError_t attn_prefill_hilo(const Dims &d, const float *Q, bf16 *o_hi, bf16 *o_lo, const TKV *kc,
                              const TKV *vc, int p0, int n, cudaStream_t st)
{
    const int hg = d.NH < 16 ? d.NH : 16;
    k_attn_prefill<float, TKV, true><<<dim3(n, (d.NH + hg - 1) / hg), 256, attn_prefill_smem(d), st>>>(
        Q, o_hi, o_lo, kc, vc, p0, d, hg);
    ++launch_count();
    return cudaGetLastError();
}
template cudaError_t attn_prefill_hilo<bf16>(const Dims &, const float *, bf16 *, bf16 *, const bf16 *,
                                             const bf16 *, int, int, cudaStream_t);
template cudaError_t attn_prefill_hilo<float>(const Dims &, const float *, bf16 *, bf16 *, const float *,
                                              const float *, int, int, cudaStream_t);

template <typename TA, typename TW, typename TKV>
static cudaError_t chunk_t(const Dims &d, const LayerPtrs *layers, void *const *kcs,
                           void *const *vcs, const float2 *rope, const uint16_t *tok_embd,
                           const PrefillBufs &pb, int p0, int n, cudaStream_t st, int nsm)
{
    cudaError_t e;
    const int H = d.H, K = d.K, nent = n * K;
    TA *XN = (TA *)pb.XN, *C = (TA *)pb.C, *Q = (TA *)pb.Q, *O = (TA *)pb.O;
    TA *HG = (TA *)pb.HG, *HS = (TA *)pb.HS;
    k_embed_rows<<<n, 256, 0, st>>>(tok_embd, pb.tok, pb.X, H);
    ++launch_count();
    if ((e = cudaGetLastError())) return e;
    for (int l = 0; l <= d.L; ++l) {
        for (int i = 0; i < pb.n_rec; ++i)
            if ((e = cudaMemcpyAsync(pb.rec_dst[i] + (size_t)l * H, pb.X + (size_t)pb.rec_row[i] * H,
                                     (size_t)H * 4, cudaMemcpyDeviceToDevice, st)))
                return e;
        if (l == d.L) break;
        const LayerPtrs &w = layers[l];
        TKV *kc = (TKV *)kcs[l], *vc = (TKV *)vcs[l];
        k_rmsnorm_rows<TA><<<n, 256, 0, st>>>(pb.X, w.attn_norm, XN, nullptr, H, d.eps);
        ++launch_count();
        ProbQKVA<TA, TW> pa{XN, (const TW *)w.wq_a, (const TW *)w.wkv_a, C, H, d.RQ, d.RQ + d.RKV};
        if ((e = gemm_dense<TA, TW>(pa, n, d.RQ + d.RKV, H, st, nsm))) return e;
        ProbQB<TA, TW> pq{C, (const TW *)w.wq_b, Q, rope, d.RQ + d.RKV, d.RQ, d.QD, d.HD, p0};
        if ((e = gemm_dense<TA, TW>(pq, n, d.QD, d.RQ, st, nsm))) return e;
        ProbKVB<TA, TW, TKV> pk{C, (const TW *)w.wk_b, (const TW *)w.wv_b, kc, vc, rope,
                                d.RQ + d.RKV, d.RQ, d.RKV, d.HD, p0};
        if ((e = gemm_dense<TA, TW>(pk, n, 2 * d.HD, d.RKV, st, nsm))) return e;
        const int hg = d.NH < 16 ? d.NH : 16;
        k_attn_prefill<TA, TKV><<<dim3(n, (d.NH + hg - 1) / hg), 256, attn_prefill_smem(d), st>>>(
            Q, O, nullptr, kc, vc, p0, d, hg);
        ++launch_count();
        if ((e = cudaGetLastError())) return e;
        ProbWO<TA, TW> po{O, (const TW *)w.wo, pb.X, d.QD, H};
        if ((e = gemm_dense<TA, TW>(po, n, H, d.QD, st, nsm))) return e;
        k_rmsnorm_rows<TA><<<n, 256, 0, st>>>(pb.X, w.ffn_norm, XN, pb.XN32, H, d.eps);
        ++launch_count();
        ProbRouter<TW> pr{pb.XN32, (const TW *)w.w_router, pb.S, H, d.E};
        if ((e = gemm_dense<float, TW>(pr, n, d.E, H, st, nsm))) return e;
        k_router_topk<<<(n * 32 + 255) / 256, 256, 0, st>>>(pb.S, 1, 0, pb.ids, pb.wts, n, d.E, K, pb.status);
        ++launch_count();
        if ((e = group_by_expert(pb, nent, d.E, kGroupBM, st))) return e;
        const int max_tiles = nent / kGroupBM + d.E + 1;
        ProbGU<TA, TW, true> pg{XN, pb.rows, (const TW *)w.w_gate, (const TW *)w.w_up, HG, H,
                                d.I, K, (size_t)d.I * H};
        if ((e = gemm_grouped<TA, TW>(pg, pb.tiles, pb.off, max_tiles, 2 * d.I, H, st))) return e;
        ProbGU<TA, TW, false> ps{XN, nullptr, (const TW *)w.ws_gate, (const TW *)w.ws_up, HS, H,
                                 d.I, K, 0};
        if ((e = gemm_dense<TA, TW>(ps, n, 2 * d.I, H, st, nsm))) return e;
        ProbDown<TA, TW> pd{HG, pb.rows, (const TW *)w.w_down, pb.YS, H, d.I};
        if ((e = gemm_grouped<TA, TW>(pd, pb.tiles, pb.off, max_tiles, H, d.I, st))) return e;
        ProbSharedDown<TA, TW> psd{HS, (const TW *)w.ws_down, pb.YS, pb.wts, pb.X, H, d.I, K};
        if ((e = gemm_dense<TA, TW>(psd, n, H, d.I, st, nsm))) return e;
    }
    return cudaGetLastError();
}

cudaError_t prefill_chunk(const Dims &d, const LayerPtrs *layers, void *const *kc,
                          void *const *vc, const float2 *rope, const uint16_t *tok_embd,
                          const PrefillBufs &pb, int p0, int n, cudaStream_t st, int nsm)
{
    // SIMT path: f32 activations for every weight format
    if (d.wdt == DS4G_BF16)
        return d.kvdt == DS4G_BF16
                   ? chunk_t<float, bf16, bf16>(d, layers, kc, vc, rope, tok_embd, pb, p0, n, st, nsm)
                   : chunk_t<float, bf16, float>(d, layers, kc, vc, rope, tok_embd, pb, p0, n, st, nsm);
    return d.kvdt == DS4G_BF16
               ? chunk_t<float, float, bf16>(d, layers, kc, vc, rope, tok_embd, pb, p0, n, st, nsm)
               : chunk_t<float, float, float>(d, layers, kc, vc, rope, tok_embd, pb, p0, n, st, nsm);
}

}  // namespace ds4g
