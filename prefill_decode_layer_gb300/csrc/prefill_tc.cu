// Layer-major prefill on the tensor cores (page "ds4.c 学习笔记 -- 端到端推理流程",
// 阶段三 prefill_layer_major_cpu: every layer runs over the whole chunk before the
// next, so each layer's weights are read once per chunk).
//
// Same steps, order and fixed reductions as the SIMT form in prefill.cu, with every
// weight contraction a tcgen05 GEMM (tc_gemm.cuh).  Activations entering a GEMM are
// stored as BF16 hi/lo pairs; the residual, the queries and the router scores stay
// FP32.  The buffers are those of the SIMT form: an FP32-sized buffer holds exactly
// one hi and one lo BF16 array, and the grouped copy of the MoE input (needed only
// by the routed gate/up GEMM) lives in the routed-output buffer, which is written
// only afterwards.  Weight tensor maps are built once per model, activation maps
// once per session.
#include "kernels.h"
#include "prefill_problems.cuh"
#include "prefill_tc.h"
#include "tc_gemm.cuh"

namespace ds4g {

// ------------------------------------------------------------------ small kernels

__device__ __forceinline__ void split_hilo(float v, bf16 &h, bf16 &l)
{
    h = __float2bfloat16_rn(v);
    l = __float2bfloat16_rn(v - __bfloat162float(h));
}

// RMSNorm of each residual row into hi/lo BF16 (one CTA per token row).
__global__ void __launch_bounds__(256) k_rmsnorm_hilo(const float *X, const float *g, bf16 *hi, bf16 *lo,
                                                      int H, float eps)
{
    __shared__ float red[32];
    const int t = blockIdx.x;
    const float *x = X + (size_t)t * H;
    float ss = 0.f;
    for (int i = threadIdx.x; i < H; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
    ss = block_sum(ss, red);
    const float inv = rsqrtf(ss / (float)H + eps);
    for (int i = threadIdx.x; i < H; i += blockDim.x) {
        bf16 h, l;
        split_hilo(x[i] * inv * g[i], h, l);
        hi[(size_t)t * H + i] = h;
        lo[(size_t)t * H + i] = l;
    }
}

// Grouped copy of the MoE input: row r <- token rows[r] / K (16-byte chunks).
__global__ void __launch_bounds__(256) k_gather_rows(const bf16 *hi, const bf16 *lo, const int *rows, int K,
                                                     int nent, int H, bf16 *ghi, bf16 *glo)
{
    const int r = blockIdx.x;
    if (r >= nent) return;
    const size_t src = (size_t)(rows[r] / K) * H, dst = (size_t)r * H;
    const int nv = H / 8;
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
        reinterpret_cast<uint4 *>(ghi + dst)[v] = reinterpret_cast<const uint4 *>(hi + src)[v];
        reinterpret_cast<uint4 *>(glo + dst)[v] = reinterpret_cast<const uint4 *>(lo + src)[v];
    }
}

// ------------------------------------------------------------------ epilogues

struct EpiHiLo {   // out[m][n..n+3] as hi/lo BF16
    bf16 *hi, *lo;
    int ld;
    __device__ void store4(int m, int n, const float (&v)[4], int) const
    {
        __align__(8) bf16 h[4], l[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) split_hilo(v[j], h[j], l[j]);
        *reinterpret_cast<uint2 *>(hi + (size_t)m * ld + n) = *reinterpret_cast<const uint2 *>(h);
        *reinterpret_cast<uint2 *>(lo + (size_t)m * ld + n) = *reinterpret_cast<const uint2 *>(l);
    }
};

struct EpiSwiGLU {   // h[m][i..i+3] = silu(gate) * up, as hi/lo BF16
    bf16 *hi, *lo;
    int ld;
    __device__ void store_gu4(int m, int i, const float (&g)[4], const float (&u)[4], int) const
    {
        __align__(8) bf16 h[4], l[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) split_hilo(silu_mul(g[j], u[j]), h[j], l[j]);
        *reinterpret_cast<uint2 *>(hi + (size_t)m * ld + i) = *reinterpret_cast<const uint2 *>(h);
        *reinterpret_cast<uint2 *>(lo + (size_t)m * ld + i) = *reinterpret_cast<const uint2 *>(l);
    }
};

// ------------------------------------------------------------------ maps and eligibility

bool tc_prefill_eligible(const Dims &d)
{
    return d.wdt == DS4G_BF16 && d.H % 128 == 0 && d.RQ % 128 == 0 && d.RKV % 128 == 0 &&
           d.QD % 128 == 0 && d.HD % 128 == 0 && d.E % 128 == 0 && d.I % 64 == 0;
}

cudaError_t tc_layer_maps(const Dims &d, const LayerPtrs &w, TcLayerMaps &m)
{
    using tc::make_map_bf16;
    const int H = d.H, I = d.I, E = d.E;
    cudaError_t e;
    if ((e = make_map_bf16(&m.wqa, w.wq_a, d.RQ, H, H, 128))) return e;
    if ((e = make_map_bf16(&m.wkva, w.wkv_a, d.RKV, H, H, 128))) return e;
    if ((e = make_map_bf16(&m.wqb, w.wq_b, d.QD, d.RQ, d.RQ, 128))) return e;
    if ((e = make_map_bf16(&m.wkb, w.wk_b, d.HD, d.RKV, d.RKV, 128))) return e;
    if ((e = make_map_bf16(&m.wvb, w.wv_b, d.HD, d.RKV, d.RKV, 128))) return e;
    if ((e = make_map_bf16(&m.wo, w.wo, H, d.QD, d.QD, 128))) return e;
    if ((e = make_map_bf16(&m.wr, w.w_router, E, H, H, 128))) return e;
    if ((e = make_map_bf16(&m.wsg, w.ws_gate, I, H, H, 64))) return e;
    if ((e = make_map_bf16(&m.wsu, w.ws_up, I, H, H, 64))) return e;
    if ((e = make_map_bf16(&m.wsd, w.ws_down, H, I, I, 128))) return e;
    if ((e = make_map_bf16(&m.wg, w.w_gate, E * I, H, H, 64))) return e;
    if ((e = make_map_bf16(&m.wu, w.w_up, E * I, H, H, 64))) return e;
    return make_map_bf16(&m.wd, w.w_down, E * H, I, I, 128);
}

TcActPtrs tc_act_ptrs(const Dims &d, const PrefillBufs &pb)
{
    const size_t P = pb.P, PK = (size_t)pb.P * d.K, RC = d.RQ + d.RKV;
    TcActPtrs a;
    a.xn_hi = (bf16 *)pb.XN;
    a.xn_lo = a.xn_hi + P * d.H;
    a.c_hi = (bf16 *)pb.C;
    a.c_lo = a.c_hi + P * RC;
    a.o_hi = (bf16 *)pb.O;
    a.o_lo = a.o_hi + P * d.QD;
    a.xg_hi = (bf16 *)pb.YS;   // dead once the routed gate/up GEMM has run
    a.xg_lo = a.xg_hi + PK * d.H;
    a.hg_hi = (bf16 *)pb.HG;
    a.hg_lo = a.hg_hi + PK * d.I;
    a.hs_hi = (bf16 *)pb.HS;
    a.hs_lo = a.hs_hi + P * d.I;
    return a;
}

cudaError_t tc_act_maps(const Dims &d, const PrefillBufs &pb, TcActMaps &m)
{
    using tc::make_map_bf16;
    const TcActPtrs a = tc_act_ptrs(d, pb);
    const int P = pb.P, PK = pb.P * d.K, RC = d.RQ + d.RKV;
    cudaError_t e;
    if ((e = make_map_bf16(&m.xn_hi, a.xn_hi, P, d.H, d.H, tc::BN))) return e;
    if ((e = make_map_bf16(&m.xn_lo, a.xn_lo, P, d.H, d.H, tc::BN))) return e;
    if ((e = make_map_bf16(&m.c_hi, a.c_hi, P, RC, RC, tc::BN))) return e;
    if ((e = make_map_bf16(&m.c_lo, a.c_lo, P, RC, RC, tc::BN))) return e;
    if ((e = make_map_bf16(&m.o_hi, a.o_hi, P, d.QD, d.QD, tc::BN))) return e;
    if ((e = make_map_bf16(&m.o_lo, a.o_lo, P, d.QD, d.QD, tc::BN))) return e;
    if ((e = make_map_bf16(&m.xg_hi, a.xg_hi, PK, d.H, d.H, tc::BN))) return e;
    if ((e = make_map_bf16(&m.xg_lo, a.xg_lo, PK, d.H, d.H, tc::BN))) return e;
    if ((e = make_map_bf16(&m.hg_hi, a.hg_hi, PK, d.I, d.I, tc::BN))) return e;
    if ((e = make_map_bf16(&m.hg_lo, a.hg_lo, PK, d.I, d.I, tc::BN))) return e;
    if ((e = make_map_bf16(&m.hs_hi, a.hs_hi, P, d.I, d.I, tc::BN))) return e;
    return make_map_bf16(&m.hs_lo, a.hs_lo, P, d.I, d.I, tc::BN);
}

// ------------------------------------------------------------------ one chunk

template <typename TKV>
static cudaError_t chunk_tc_t(const Dims &d, const LayerPtrs *layers, const TcLayerMaps *lm,
                              const TcActMaps &am, void *const *kcs, void *const *vcs, const float2 *rope,
                              const uint16_t *tok_embd, const PrefillBufs &pb, int p0, int n,
                              cudaStream_t st)
{
    cudaError_t e;
    const int H = d.H, K = d.K, nent = n * K, I = d.I;
    const TcActPtrs ap = tc_act_ptrs(d, pb);
    const int ny = (n + tc::BN - 1) / tc::BN;
    const int max_tiles = nent / tc::BN + d.E + 1;
    tc::Args a{};
    a.status = pb.status;
    k_embed_rows<<<n, 256, 0, st>>>(tok_embd, pb.tok, pb.X, H);
    ++launch_count();
    if ((e = cudaGetLastError())) return e;
    for (int l = 0; l < d.L; ++l) {
        const LayerPtrs &w = layers[l];
        const TcLayerMaps &m = lm[l];
        TKV *kc = (TKV *)kcs[l], *vc = (TKV *)vcs[l];
        // attention half
        k_rmsnorm_hilo<<<n, 256, 0, st>>>(pb.X, w.attn_norm, ap.xn_hi, ap.xn_lo, H, d.eps);
        ++launch_count();
        a = tc::Args{};
        a.status = pb.status;
        a.m_tok = n;
        a.n_out = d.RQ + d.RKV, a.k = H, a.piece_rows = d.RQ;
        if ((e = tc::launch<false>(m.wqa, m.wkva, am.xn_hi, am.xn_lo, a,
                                   EpiHiLo{ap.c_hi, ap.c_lo, d.RQ + d.RKV}, (d.RQ + d.RKV) / tc::BM, ny, st)))
            return e;
        a.n_out = d.QD, a.k = d.RQ, a.piece_rows = 0, a.x_col0 = 0;
        ProbQB<float, bf16> pq{nullptr, nullptr, (float *)pb.Q, rope, 0, d.RQ, d.QD, d.HD, p0};
        if ((e = tc::launch<false>(m.wqb, m.wqb, am.c_hi, am.c_lo, a, pq, d.QD / tc::BM, ny, st))) return e;
        a.n_out = 2 * d.HD, a.k = d.RKV, a.piece_rows = d.HD, a.x_col0 = d.RQ;
        ProbKVB<float, bf16, TKV> pk{nullptr, nullptr, nullptr, kc, vc, rope, 0, d.RQ, d.RKV, d.HD, p0};
        if ((e = tc::launch<false>(m.wkb, m.wvb, am.c_hi, am.c_lo, a, pk, 2 * d.HD / tc::BM, ny, st))) return e;
        if ((e = attn_prefill_hilo<TKV>(d, (const float *)pb.Q, ap.o_hi, ap.o_lo, kc, vc, p0, n, st))) return e;
        a.n_out = H, a.k = d.QD, a.piece_rows = 0, a.x_col0 = 0;
        ProbWO<float, bf16> po{nullptr, nullptr, pb.X, d.QD, H};
        if ((e = tc::launch<false>(m.wo, m.wo, am.o_hi, am.o_lo, a, po, H / tc::BM, ny, st))) return e;
        // MoE half
        k_rmsnorm_hilo<<<n, 256, 0, st>>>(pb.X, w.ffn_norm, ap.xn_hi, ap.xn_lo, H, d.eps);
        ++launch_count();
        a.n_out = d.E, a.k = H;
        ProbRouter<bf16> pr{nullptr, nullptr, pb.S, H, d.E};
        if ((e = tc::launch<false>(m.wr, m.wr, am.xn_hi, am.xn_lo, a, pr, d.E / tc::BM, ny, st))) return e;
        k_router_topk<<<(n * 32 + 255) / 256, 256, 0, st>>>(pb.S, pb.ids, pb.wts, n, d.E, K, pb.status);
        ++launch_count();
        k_group_count<<<d.E, 256, 0, st>>>(pb.ids, nent, pb.cnt);
        ++launch_count();
        k_group_scan<<<1, 32, 0, st>>>(pb.cnt, d.E, tc::BN, pb.off, pb.tiles);
        ++launch_count();
        k_group_fill<<<d.E, 256, 0, st>>>(pb.ids, nent, pb.off, pb.rows);
        ++launch_count();
        k_gather_rows<<<nent, 256, 0, st>>>(ap.xn_hi, ap.xn_lo, pb.rows, K, nent, H, ap.xg_hi, ap.xg_lo);
        ++launch_count();
        if ((e = cudaGetLastError())) return e;
        // routed gate/up + SwiGLU (grouped), then the shared expert's
        tc::Args g{};
        g.status = pb.status;
        g.n_out = I, g.k = H, g.tiles = pb.tiles, g.off = pb.off;
        if ((e = tc::launch<true>(m.wg, m.wu, am.xg_hi, am.xg_lo, g, EpiSwiGLU{ap.hg_hi, ap.hg_lo, I},
                                  I / (tc::BM / 2), max_tiles, st)))
            return e;
        a.n_out = I, a.k = H;
        if ((e = tc::launch<true>(m.wsg, m.wsu, am.xn_hi, am.xn_lo, a, EpiSwiGLU{ap.hs_hi, ap.hs_lo, I},
                                  I / (tc::BM / 2), ny, st)))
            return e;
        // routed down (grouped) into per-(token, slot) rows, then the shared down
        // projection whose epilogue adds the weighted routed rows and the residual
        g.n_out = H, g.k = I;
        ProbDown<float, bf16> pd{nullptr, pb.rows, nullptr, pb.YS, H, I};
        if ((e = tc::launch<false>(m.wd, m.wd, am.hg_hi, am.hg_lo, g, pd, H / tc::BM, max_tiles, st))) return e;
        a.n_out = H, a.k = I;
        ProbSharedDown<float, bf16> psd{nullptr, nullptr, pb.YS, pb.wts, pb.X, H, I, K};
        if ((e = tc::launch<false>(m.wsd, m.wsd, am.hs_hi, am.hs_lo, a, psd, H / tc::BM, ny, st))) return e;
    }
    return cudaGetLastError();
}

cudaError_t prefill_chunk_tc(const Dims &d, const LayerPtrs *layers, const TcLayerMaps *lm,
                             const TcActMaps &am, void *const *kc, void *const *vc, const float2 *rope,
                             const uint16_t *tok_embd, const PrefillBufs &pb, int p0, int n, cudaStream_t st)
{
    return d.kvdt == DS4G_BF16 ? chunk_tc_t<bf16>(d, layers, lm, am, kc, vc, rope, tok_embd, pb, p0, n, st)
                               : chunk_tc_t<float>(d, layers, lm, am, kc, vc, rope, tok_embd, pb, p0, n, st);
}

}  // namespace ds4g
