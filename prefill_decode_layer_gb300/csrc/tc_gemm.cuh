// Tensor-core GEMM for the layer-major prefill (sm_103a, tcgen05 + TMA).
//
//   out[token][n] = sum_k W[n][k] * (Xhi[token][k] + Xlo[token][k])
//
// W is a BF16 weight matrix ([out][in], K contiguous).  The activations are
// carried as two BF16 arrays: hi = bf16(x) and lo = bf16(x - hi), so that every
// product is taken with about 16 significant bits of x and accumulated in FP32.
// With single BF16 activations the prefill's hidden states drift by about 0.5 %
// per layer, which flips router top-6 decisions (the 6th-to-7th score gaps are
// small); the split keeps the decisions of an FP32 computation.
//
// Orientation: the weight rows are the MMA's M side (128 rows per tile) and the
// tokens its N side (128 per tile), so a tile of W is multiplied with the hi and
// the lo tile of the same tokens: two MMAs per 16-wide K step into one FP32
// accumulator in tensor memory (128 lanes x 128 columns).  A tile that owns fewer
// than 128 token rows (an expert's last rows, a ragged chunk) runs its MMAs with N
// = its rows rounded up to 16.
//
// Persistent: one CTA per SM walks the output tiles (weight-row block fastest, so
// CTAs running together share a token tile in L2) with 192 threads:
//   warp 0 lane 0   TMA producer: per 64-wide K stage, the W tile (16 KB) and the
//                   hi and lo token tiles (16 KB each), 128-byte swizzled, into a
//                   4-stage shared-memory ring (full / empty mbarriers) that runs
//                   on across tile boundaries;
//   warp 1          allocates two accumulators in TMEM (2 x 128 columns); lane 0
//                   issues the MMAs of tile i into accumulator i % 2 as soon as the
//                   epilogue has drained it, and commits each stage back to the
//                   producer and each tile to the epilogue;
//   warps 2-5       epilogue, overlapping the next tile's MMAs: TMEM -> registers ->
//                   a [token][feature] FP32 half tile in shared memory -> the
//                   problem's functor, four adjacent features at a time, so RoPE
//                   pairs are local to one call; a functor's global loads (load4)
//                   are issued eight at a time before the matching stores.
// Gate/up tiles (GU) hold 128 gate rows and the same 128 up rows in two
// accumulators that share each token tile; SwiGLU is applied straight from the
// two accumulators (a feature's gate and up sit in the same TMEM lane).
// Every wait is bounded; a CTA that gives up raises DS4G_ETIMEOUT in *status, lets
// its MMAs and copies finish, frees its TMEM and returns.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "sm100.cuh"

namespace ds4g {
namespace tc {

static constexpr int BM = 128;      // weight rows per accumulator (MMA M)
static constexpr int BN = 128;      // tokens per tile (MMA N)
static constexpr int BK = 64;       // K per stage: one 128-byte swizzle row of BF16
static constexpr int THREADS = 192;
static constexpr uint32_t TILE_A = BM * BK * 2;              // 16 KB
static constexpr uint32_t TILE_B = BN * BK * 2;              // 16 KB
static constexpr int HALF = BN / 2;                          // tokens staged at once
static constexpr int EPI_PITCH = BM + 4;                     // floats per staged token row
static constexpr uint32_t EPI_BYTES = HALF * EPI_PITCH * 4;  // 33 KB
static constexpr int EPI_BATCH = 8;                          // functor loads in flight

// Tile geometry.  Plain: 128 weight rows, one accumulator, 4 stages of 48 KB and a
// staged epilogue.  Gate/up (GU): 128 gate rows and the same 128 up rows, two
// accumulators sharing every token tile (the activations are read half as often),
// 3 stages of 64 KB, and SwiGLU straight from the two accumulators.
template <bool GU> struct Geo {
    static constexpr int NACC = GU ? 2 : 1;
    static constexpr uint32_t XOFF = NACC * TILE_A;          // token tiles after the W tiles
    static constexpr uint32_t STAGE = XOFF + 2 * TILE_B;
    static constexpr int STAGES = GU ? 3 : 4;
    static constexpr uint32_t TMEM_COLS = 2 * NACC * BN;     // two tiles in flight
    static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE + (GU ? 0 : EPI_BYTES) + 256;
};

// What a launch computes.  Dense: token rows [0, m_tok) in tiles of BN.  Grouped
// (tiles != nullptr): token tile j is (expert e, first grouped row r0) from the
// tile list, rows [r0, off[e+1]) of the grouped activations, and expert e's weight
// rows start at e * n_out.  Weight-row blocks: n_out / BM (for GU, n_out is the
// number of gate rows = up rows).
struct Args {
    int n_out;        // weight rows (per expert when grouped)
    int k;            // reduction length, a multiple of BK
    int x_col0;       // first activation column read (a multiple of 8)
    int piece_rows;   // dense: rows of map w0 before map w1 starts (0: w0 only)
    int m_tok;        // dense: token rows
    const int *tiles; // grouped: [0] = count, then (expert, first row) pairs
    const int *off;   // grouped: expert row offsets [E + 1]
    int *status;      // DS4G_ETIMEOUT on a wait that gave up
};

struct NoAux {};

// GU: the tile's gate rows come from w0 and its up rows from w1 (same row index);
// the epilogue calls Epi::store_h(m, i, silu(gate) * up, e) per element.
// Otherwise Epi provides  Aux load4(m, n, e)  and  store4(m, n, v[4], aux, e).
template <class Epi, bool GU>
__global__ void __launch_bounds__(THREADS, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap w0, const __grid_constant__ CUtensorMap w1,
              const __grid_constant__ CUtensorMap xhi, const __grid_constant__ CUtensorMap xlo,
              const Args a, const Epi epi)
{
    using G = Geo<GU>;
    constexpr int STAGES = G::STAGES;
    constexpr uint32_t STAGE_BYTES = G::STAGE;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float *stg = reinterpret_cast<float *>(sm + STAGES * STAGE_BYTES);   // [HALF][EPI_PITCH] (plain)
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + STAGES * STAGE_BYTES + (GU ? 0 : EPI_BYTES));
    uint64_t *empty = full + STAGES;
    uint64_t *accf = empty + STAGES;   // [2] accumulator ready (MMA commit)
    uint64_t *acce = accf + 2;         // [2] accumulator drained (128 epilogue threads)
    uint64_t *done = acce + 2;         // every MMA of this CTA completed
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);
    int *abort_flag = reinterpret_cast<int *>(tslot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int mtiles = a.n_out / BM;
    const int ntiles = a.tiles ? a.tiles[0] : (a.m_tok + BN - 1) / BN;
    const int total = mtiles * ntiles;
    const int nk = a.k / BK;
    // tile -> (weight block mb, expert e, first token row r0, end row)
    auto tile_of = [&](int tau, int &mb, int &e, int &r0, int &rend) {
        mb = tau % mtiles;
        const int j = tau / mtiles;
        if (a.tiles) {
            e = a.tiles[1 + 2 * j];
            r0 = a.tiles[2 + 2 * j];
            rend = min(r0 + BN, a.off[e + 1]);
        } else {
            e = 0;
            r0 = j * BN;
            rend = min(r0 + BN, a.m_tok);
        }
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 128);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(tslot, G::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    volatile int *ab = abort_flag;
    auto give_up = [&]() {
        *abort_flag = 1;
        atomicExch(a.status, DS4G_ETIMEOUT);
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            tma_prefetch_desc(&w0);
            tma_prefetch_desc(&w1);
            tma_prefetch_desc(&xhi);
            tma_prefetch_desc(&xlo);
            unsigned it = 0;
            bool ok = true;
            for (int tau = blockIdx.x; ok && tau < total; tau += gridDim.x) {
                int mb, e, r0, rend;
                tile_of(tau, mb, e, r0, rend);
                const void *wm = &w0;
                int wrow;
                if (GU) {
                    wrow = e * a.n_out + mb * BM;
                } else if (a.piece_rows > 0 && mb * BM >= a.piece_rows) {
                    wm = &w1;
                    wrow = mb * BM - a.piece_rows;
                } else {
                    wrow = e * a.n_out + mb * BM;
                }
                for (int i = 0; i < nk; ++i, ++it) {
                    const int s = it % STAGES;
                    if (!mbar_wait(&empty[s], ((it / STAGES) & 1) ^ 1, ab)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    unsigned char *st = sm + s * STAGE_BYTES;
                    mbar_expect_tx(&full[s], STAGE_BYTES);
                    const int kx = i * BK;
                    if (GU) {
                        tma_load_2d(st, &w0, kx, wrow, &full[s]);
                        tma_load_2d(st + TILE_A, &w1, kx, wrow, &full[s]);
                    } else {
                        tma_load_2d(st, wm, kx, wrow, &full[s]);
                    }
                    tma_load_2d(st + G::XOFF, &xhi, a.x_col0 + kx, r0, &full[s]);
                    tma_load_2d(st + G::XOFF + TILE_B, &xlo, a.x_col0 + kx, r0, &full[s]);
                }
            }
            // no copy may still be in flight when the CTA exits
            const unsigned n = it < (unsigned)STAGES ? it : (unsigned)STAGES;
            for (unsigned q = 1; q <= n; ++q) {
                const unsigned i = it - q;
                volatile int never = 0;
                mbar_wait(&full[i % STAGES], (i / STAGES) & 1, &never);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            unsigned it = 0, tc = 0;
            bool ok = true;
            for (int tau = blockIdx.x; ok && tau < total; tau += gridDim.x, ++tc) {
                const int b = tc & 1;
                // MMA N: the tile's token rows rounded up to 16 (a ragged or grouped
                // tile skips the rows it does not own; their columns are never read)
                int mb, e, r0, rend;
                tile_of(tau, mb, e, r0, rend);
                const int nn = min(BN, max(16, (rend - r0 + 15) & ~15));
                const uint32_t idesc = idesc_bf16_f32(BM, nn);
                if (!mbar_wait(&acce[b], ((tc >> 1) & 1) ^ 1, ab)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(b * G::NACC * BN);
                for (int i = 0; i < nk; ++i, ++it) {
                    const int s = it % STAGES;
                    if (!mbar_wait(&full[s], (it / STAGES) & 1, ab)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(sm + s * STAGE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t bh = sdesc_kmajor_sw128(sa + G::XOFF + kk * 32);
                        const uint64_t bl = sdesc_kmajor_sw128(sa + G::XOFF + TILE_B + kk * 32);
#pragma unroll
                        for (int r = 0; r < G::NACC; ++r) {   // gate (and up) accumulators
                            const uint64_t ad = sdesc_kmajor_sw128(sa + r * TILE_A + kk * 32);
                            tc_mma_bf16(acc + r * BN, ad, bh, idesc, (i | kk) != 0);
                            tc_mma_bf16(acc + r * BN, ad, bl, idesc, 1u);
                        }
                    }
                    tc_commit(&empty[s]);   // the stage is free once these MMAs complete
                }
                if (ok) tc_commit(&accf[b]);   // the tile is complete once every MMA is
            }
            // TMEM may be freed only after every MMA issued here has completed
            tc_commit(done);
            volatile int never = 0;
            mbar_wait(done, 0, &never);
        }
    } else {
        // ---------------- epilogue (warps 2-5)
        const int q = warp & 3;            // TMEM lane quarter this warp may access
        const int et = threadIdx.x - 64;   // 0..127
        unsigned tc = 0;
        for (int tau = blockIdx.x; tau < total; tau += gridDim.x, ++tc) {
            int mb, e, r0, rend;
            tile_of(tau, mb, e, r0, rend);
            const int b = tc & 1;
            if (!mbar_wait(&accf[b], (tc >> 1) & 1, ab)) {
                give_up();
                break;
            }
            tc_fence_after();
            if constexpr (GU) {
                // gate and up of feature f = this thread's lane, 32 tokens at a time
                const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * 2 * BN);
                const int i = mb * BM + 32 * q + lane;
                const int last = max(0, ((rend - r0 - 1) >> 5) << 5);   // first column of the last chunk read
#pragma unroll 1
                for (int c0 = 0; c0 <= last; c0 += 32) {
                    float g[32], u[32];
                    tmem_ld32(lane_base + (uint32_t)c0, g);
                    tmem_ld32(lane_base + (uint32_t)(BN + c0), u);
                    if (c0 == last) {   // the accumulators are drained
                        tc_fence_before();
                        mbar_arrive(&acce[b]);
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {   // static indices keep g, u in registers
                        const int m = r0 + c0 + j;
                        if (m < rend) epi.store_h(m, i, silu_mul(g[j], u[j]), e);
                    }
                }
            } else {
            for (int h = 0; h < 2; ++h) {
                // accumulator columns (tokens) h*HALF .. +HALF-1 into stg[token][feature]
#pragma unroll 1
                for (int c0 = 0; c0 < HALF; c0 += 32) {
                    float v[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * BN + h * HALF + c0), v);
                    const int f = 32 * q + lane;
#pragma unroll
                    for (int j = 0; j < 32; ++j) stg[(c0 + j) * EPI_PITCH + f] = v[j];
                }
                if (h == 1) {   // the accumulator is drained: the next tile may use it
                    tc_fence_before();
                    mbar_arrive(&acce[b]);
                }
                asm volatile("bar.sync 2, 128;" ::: "memory");
                const int tbase = r0 + h * HALF;
                {
                    constexpr int NI = HALF * (BM / 4) / 128;   // items per thread (16)
#pragma unroll 1
                    for (int i0 = 0; i0 < NI; i0 += EPI_BATCH) {
                        typename Epi::Aux aux[EPI_BATCH];
#pragma unroll
                        for (int u = 0; u < EPI_BATCH; ++u) {
                            const int idx = et + 128 * (i0 + u);
                            const int t = idx / (BM / 4), j = (idx % (BM / 4)) * 4;
                            if (tbase + t < rend) aux[u] = epi.load4(tbase + t, mb * BM + j, e);
                        }
#pragma unroll
                        for (int u = 0; u < EPI_BATCH; ++u) {
                            const int idx = et + 128 * (i0 + u);
                            const int t = idx / (BM / 4), j = (idx % (BM / 4)) * 4;
                            if (tbase + t >= rend) continue;
                            const float4 v4 = *reinterpret_cast<const float4 *>(stg + t * EPI_PITCH + j);
                            const float v[4] = {v4.x, v4.y, v4.z, v4.w};
                            epi.store4(tbase + t, mb * BM + j, v, aux[u], e);
                        }
                    }
                }
                asm volatile("bar.sync 2, 128;" ::: "memory");   // stg is rewritten next
            }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, G::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side

// Tensor map of a row-major BF16 matrix [rows][cols] (row stride ld elements) read
// in boxes of 64 columns x box_rows rows with the 128-byte swizzle; rows beyond
// `rows` read as zeros.
cudaError_t make_map_bf16(CUtensorMap *m, const void *base, int rows, int cols, int ld, int box_rows);

// ntile_bound: token tiles at most (dense: exact; grouped: the tile list's bound).
template <bool GU, class Epi>
static cudaError_t launch(const CUtensorMap &w0, const CUtensorMap &w1, const CUtensorMap &xhi,
                          const CUtensorMap &xlo, const Args &a, const Epi &epi, int mtiles, int ntile_bound,
                          int nsm, cudaStream_t st)
{
    const long long work = (long long)mtiles * ntile_bound;
    if (work <= 0) return cudaSuccess;
    static bool attr_set = false;   // per instantiation; set before the first launch
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_tc_gemm<Epi, GU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)Geo<GU>::SMEM);
        if (e) return e;
        attr_set = true;
    }
    const int grid = (int)(work < nsm ? work : nsm);
    k_tc_gemm<Epi, GU><<<grid, THREADS, Geo<GU>::SMEM, st>>>(w0, w1, xhi, xlo, a, epi);
    ++launch_count();
    return cudaGetLastError();
}

}  // namespace tc
}  // namespace ds4g
