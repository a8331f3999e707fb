// Tiled SIMT GEMM over "problem" descriptors: out = A W^T with A rows and W rows
// supplied by the problem (dense, gathered or per-expert), fp32 accumulation in
// k order, and an epilogue that receives four adjacent output columns at once
// (so RoPE pairs and gate/up pairs are local to one call).
#pragma once

#include "common.cuh"

namespace ds4g {

static constexpr int kGroupBM = 64;  // rows per grouped tile (one expert per tile)

template <typename TA, typename TW, class Prob, bool GROUPED>
__global__ void __launch_bounds__(256) k_gemm_simt(Prob pb, int M, int N, int K,
                                                   const int *tiles, const int *off)
{
    constexpr int BM = 64, BN = 64, BK = 32;
    __shared__ float As[BK][BM + 4];
    __shared__ float Ws[BK][BN + 4];
    int m0, mend, g = 0;
    if constexpr (GROUPED) {
        const int t = blockIdx.y;
        if (t >= tiles[0]) return;
        g = tiles[1 + 2 * t];
        m0 = tiles[2 + 2 * t];
        mend = min(m0 + BM, off[g + 1]);
    } else {
        m0 = blockIdx.y * BM;
        mend = min(m0 + BM, M);
    }
    const int n0 = blockIdx.x * BN;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int lk = tid & 31, lr = tid >> 5;
    const TA *arow[8];
    const TW *wrow[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int m = m0 + lr + 8 * i, n = n0 + lr + 8 * i;
        arow[i] = m < mend ? pb.a_row(m, g) : nullptr;
        wrow[i] = n < N ? pb.w_row(n, g) : nullptr;
    }
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int k0 = 0; k0 < K; k0 += BK) {
        const int k = k0 + lk;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            As[lk][lr + 8 * i] = (arow[i] && k < K) ? to_f32<TA>(arow[i][k]) : 0.f;
            Ws[lk][lr + 8 * i] = (wrow[i] && k < K) ? to_f32<TW>(wrow[i][k]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < BK; ++kk) {
            const float4 a = *reinterpret_cast<const float4 *>(&As[kk][ty * 4]);
            const float4 w = *reinterpret_cast<const float4 *>(&Ws[kk][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w}, wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], wv[j], acc[i][j]);
        }
        __syncthreads();
    }
    const int n = n0 + tx * 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m < mend && n < N) pb.store4(m, n, acc[i], g);
    }
}

// out rows [0, M): grid over 64 x 64 tiles.  N must be a multiple of 4.
template <typename TA, typename TW, class Prob>
static cudaError_t gemm_dense(const Prob &pb, int M, int N, int K, cudaStream_t st, int nsm)
{
    (void)nsm;
    if (M <= 0) return cudaSuccess;
    const dim3 grid((N + 63) / 64, (M + 63) / 64);
    k_gemm_simt<TA, TW, Prob, false><<<grid, 256, 0, st>>>(pb, M, N, K, nullptr, nullptr);
    ++launch_count();
    return cudaGetLastError();
}

// Rows grouped per expert: tiles[0] work items (expert, first row), each at most
// kGroupBM rows and never crossing an expert boundary (off[e+1]).
template <typename TA, typename TW, class Prob>
static cudaError_t gemm_grouped(const Prob &pb, const int *tiles, const int *off, int max_tiles,
                                int N, int K, cudaStream_t st)
{
    const dim3 grid((N + 63) / 64, max_tiles);
    k_gemm_simt<TA, TW, Prob, true><<<grid, 256, 0, st>>>(pb, 0, N, K, tiles, off);
    ++launch_count();
    return cudaGetLastError();
}

}  // namespace ds4g
