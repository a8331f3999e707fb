// Output problems of the prefill GEMMs: which rows of A and W a SIMT tile reads
// (a_row, w_row) and what the epilogue does with four adjacent output columns of
// one row (store4).  The tensor-core GEMM (prefill_tc.cu) reuses the epilogues.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace ds4g {

// Each problem maps rows of A, rows of W (an [N][K] row-major operand) and a 4-wide
// column group of outputs; see gemm.cuh for the kernels that drive them.

template <typename TA, typename TW>
struct ProbQKVA {  // C = XN [W_qa; W_kva]^T
    const TA *XN; const TW *wqa, *wkva; TA *C; int H, RQ, ldc;
    __device__ const TA *a_row(int m, int) const { return XN + (size_t)m * H; }
    __device__ const TW *w_row(int n, int) const {
        return n < RQ ? wqa + (size_t)n * H : wkva + (size_t)(n - RQ) * H;
    }
    __device__ void store4(int m, int n, const float (&v)[4], int) const {
#pragma unroll
        for (int j = 0; j < 4; ++j) C[(size_t)m * ldc + n + j] = from_f32<TA>(v[j]);
    }
};

template <typename TA, typename TW>
struct ProbQB {  // Q = RoPE(C[:, :RQ] W_qb^T)
    const TA *C; const TW *wqb; TA *Q; const float2 *rope; int ldc, RQ, QD, HD, p0;
    __device__ const TA *a_row(int m, int) const { return C + (size_t)m * ldc; }
    __device__ const TW *w_row(int n, int) const { return wqb + (size_t)n * RQ; }
    __device__ void store4(int m, int n, const float (&v)[4], int) const {
        // two RoPE pairs: (cos, sin) of pair (n % HD) / 2 and the next, one 16-byte load
        const float4 cs = *reinterpret_cast<const float4 *>(rope + (size_t)(p0 + m) * (HD / 2) + (n % HD) / 2);
        const float r0 = v[0] * cs.x - v[1] * cs.y, r1 = v[0] * cs.y + v[1] * cs.x;
        const float r2 = v[2] * cs.z - v[3] * cs.w, r3 = v[2] * cs.w + v[3] * cs.z;
        if constexpr (std::is_same<TA, float>::value) {
            *reinterpret_cast<float4 *>(Q + (size_t)m * QD + n) = make_float4(r0, r1, r2, r3);
        } else {
            Q[(size_t)m * QD + n] = from_f32<TA>(r0);
            Q[(size_t)m * QD + n + 1] = from_f32<TA>(r1);
            Q[(size_t)m * QD + n + 2] = from_f32<TA>(r2);
            Q[(size_t)m * QD + n + 3] = from_f32<TA>(r3);
        }
    }
};

template <typename TA, typename TW, typename TKV>
struct ProbKVB {  // K = RoPE(C[:, RQ:] W_kb^T), V = C[:, RQ:] W_vb^T, appended to the cache
    const TA *C; const TW *wkb, *wvb; TKV *kc, *vc; const float2 *rope; int ldc, RQ, RKV, HD, p0;
    __device__ const TA *a_row(int m, int) const { return C + (size_t)m * ldc + RQ; }
    __device__ const TW *w_row(int n, int) const {
        return n < HD ? wkb + (size_t)n * RKV : wvb + (size_t)(n - HD) * RKV;
    }
    __device__ void store4(int m, int n, const float (&v)[4], int) const {
        const size_t row = (size_t)(p0 + m) * HD;
        if (n < HD) {
            const float2 *rp = rope + (size_t)(p0 + m) * (HD / 2);
#pragma unroll
            for (int j = 0; j < 4; j += 2) {
                const float2 cs = rp[(n + j) / 2];
                kc[row + n + j] = from_f32<TKV>(v[j] * cs.x - v[j + 1] * cs.y);
                kc[row + n + j + 1] = from_f32<TKV>(v[j] * cs.y + v[j + 1] * cs.x);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) vc[row + n - HD + j] = from_f32<TKV>(v[j]);
        }
    }
};

template <typename TA, typename TW>
struct ProbWO {  // X += O W_o^T
    const TA *O; const TW *wo; float *X; int QD, H;
    __device__ const TA *a_row(int m, int) const { return O + (size_t)m * QD; }
    __device__ const TW *w_row(int n, int) const { return wo + (size_t)n * QD; }
    __device__ void store4(int m, int n, const float (&v)[4], int) const {
        float4 *x = reinterpret_cast<float4 *>(X + (size_t)m * H + n);
        float4 r = *x;
        r.x += v[0]; r.y += v[1]; r.z += v[2]; r.w += v[3];
        *x = r;
    }
};

template <typename TW>
struct ProbRouter {  // S = XN W_r^T from f32 activations (f32 scores)
    const float *XN; const TW *wr; float *S; int H, E;
    __device__ const float *a_row(int m, int) const { return XN + (size_t)m * H; }
    __device__ const TW *w_row(int n, int) const { return wr + (size_t)n * H; }
    __device__ void store4(int m, int n, const float (&v)[4], int) const {
#pragma unroll
        for (int j = 0; j < 4; ++j) S[(size_t)m * E + n + j] = v[j];
    }
};


// Gate/up with SwiGLU; W rows interleaved (gate_i, up_i) so an output pair is local.
template <typename TA, typename TW, bool GROUPED>
struct ProbGU {
    const TA *XN; const int *rows; const TW *wg, *wu; TA *Hout; int H, I, K;
    size_t estride;  // elements between experts' matrices (I * H)
    __device__ const TA *a_row(int m, int) const {
        return XN + (size_t)(GROUPED ? rows[m] / K : m) * H;
    }
    __device__ const TW *w_row(int n, int e) const {
        const TW *b = (n & 1) ? wu : wg;
        return b + (GROUPED ? (size_t)e * estride : 0) + (size_t)(n >> 1) * H;
    }
    __device__ void store4(int m, int n, const float (&v)[4], int) const {
        Hout[(size_t)m * I + (n >> 1)] = from_f32<TA>(silu_mul(v[0], v[1]));
        Hout[(size_t)m * I + (n >> 1) + 1] = from_f32<TA>(silu_mul(v[2], v[3]));
    }
};

template <typename TA, typename TW>
struct ProbDown {  // YS[token*K + slot] = HG W_d(e)^T, grouped rows
    const TA *HG; const int *rows; const TW *wd; float *YS; int H, I;
    __device__ const TA *a_row(int m, int) const { return HG + (size_t)m * I; }
    __device__ const TW *w_row(int n, int e) const {
        return wd + (size_t)e * H * I + (size_t)n * I;
    }
    __device__ void store4(int m, int n, const float (&v)[4], int) const {
        *reinterpret_cast<float4 *>(YS + (size_t)rows[m] * H + n) = make_float4(v[0], v[1], v[2], v[3]);
    }
};

template <typename TA, typename TW>
struct ProbSharedDown {  // X += HS W_sd^T + sum_s w[s] YS[token, s]  (slot order, then shared)
    const TA *HS; const TW *wsd; const float *YS; const float *wts; float *X; int H, I, K;
    __device__ const TA *a_row(int m, int) const { return HS + (size_t)m * I; }
    __device__ const TW *w_row(int n, int) const { return wsd + (size_t)n * I; }
    __device__ void store4(int m, int n, const float (&v)[4], int) const {
        float r[4] = {0.f, 0.f, 0.f, 0.f};
        for (int s = 0; s < K; ++s) {
            const float w = wts[(size_t)m * K + s];
            const float4 y = *reinterpret_cast<const float4 *>(YS + ((size_t)m * K + s) * H + n);
            r[0] = fmaf(w, y.x, r[0]);
            r[1] = fmaf(w, y.y, r[1]);
            r[2] = fmaf(w, y.z, r[2]);
            r[3] = fmaf(w, y.w, r[3]);
        }
        float4 *x = reinterpret_cast<float4 *>(X + (size_t)m * H + n);
        float4 o = *x;
        o.x += r[0] + v[0]; o.y += r[1] + v[1]; o.z += r[2] + v[2]; o.w += r[3] + v[3];
        *x = o;
    }
};

}  // namespace ds4g
