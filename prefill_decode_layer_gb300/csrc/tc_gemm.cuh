// Tensor-core GEMM for the layer-major prefill (sm_103a, tcgen05 + TMA).
//
//   out[token][n] = sum_k X[token][k] * W[n][k]
//
// W is a BF16 weight matrix ([out][in], K contiguous) and X BF16 activations;
// products accumulate in FP32.  With LO the activations are carried as two BF16
// arrays, hi = bf16(x) and lo = bf16(x - hi), and X = hi + lo: every product is
// then taken with about 16 significant bits of x (two MMAs per K step into the
// same accumulator).  The router's GEMM uses the pair, so that its top-6
// decisions are those of an FP32 computation outside the rounding band.
//
// Orientation: 128 tokens are the MMA's M side and WN weight rows (256, or 128 for
// GEMMs with few output tiles) its N side.  With the weights on the wide side,
// every byte the tensor core reads from shared memory feeds twice the products of
// a 128 x 128 tile; shared-memory bandwidth, not the tensor pipe, bounds the dense
// GEMMs, and the weight stream from HBM bounds the routed ones.
//
// Persistent: one CTA per SM walks the output tiles (weight block fastest, so CTAs
// running together share a token tile in L2) with 320 threads:
//   warp 0 lane 0   TMA producer: per 64-wide K stage, the weight tile (WN rows, as
//                   128-row boxes) and the token tile (16 KB; hi and lo with LO),
//                   128-byte swizzled, into a shared-memory ring (full / empty
//                   mbarriers) that runs on across tile boundaries;
//   warp 1          allocates two accumulators in TMEM (2 x WN columns); lane 0
//                   issues the MMAs of tile i into accumulator i % 2 as soon as the
//                   epilogue has drained it, and commits each stage back to the
//                   producer and each tile to the epilogue;
//   warps 2-9       epilogue, overlapping the next tile's MMAs.  Warp w reads TMEM
//                   lanes 32 (w % 4).. (its 32 tokens) and every other 32-feature
//                   chunk.  Direct form: each thread hands the problem's functor the
//                   chunk's 32 adjacent features of its token (RoPE pairs local,
//                   16-byte stores).  Staged form: the chunk goes through the warp's
//                   shared-memory rows and the functor gets four adjacent features of
//                   one token at a time, an instruction covering 4 tokens x 32
//                   features.  A functor's global loads depend on the tile's
//                   coordinates only: the first chunk's are issued before the
//                   accumulator is ready, each later chunk's while the previous chunk
//                   is stored.
// Gate/up tiles (GU): the weight tile is 128 gate rows followed by the same 128 up
// rows, so a feature's gate and up sit in the same TMEM lane, 128 columns apart;
// SwiGLU is applied straight from the accumulator and each thread writes 32
// adjacent outputs of its token.
// Every wait is bounded; a CTA that gives up raises DS4G_ETIMEOUT in *status, lets
// its MMAs and copies finish, frees its TMEM and returns.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "sm100.cuh"

namespace ds4g {
namespace tc {

static constexpr int BT = 128;      // tokens per tile (MMA M)
static constexpr int BK = 64;       // K per stage: one 128-byte swizzle row of BF16
static constexpr int BOXW = 128;    // weight rows per TMA box
static constexpr int THREADS = 320;   // producer warp, MMA warp, 8 epilogue warps
static constexpr int GWARPS = 2;      // token-row gather warps (grouped GEMMs that gather)
static constexpr int THREADS_GA = THREADS + 32 * GWARPS;
static constexpr uint32_t TILE_X = BT * BK * 2;              // 16 KB
static constexpr uint32_t BOX_BYTES = BOXW * BK * 2;         // 16 KB
static constexpr int CH = 32;                                // features per epilogue chunk
static constexpr uint32_t EPI_BYTES = 8 * 32 * CH * 4;       // 32 KB: [8 warps][32 tokens][CH]
static constexpr int EPI_BATCH = 8;                          // functor loads in flight (staged)
static constexpr size_t SMEM_MAX = 232448;                   // shared memory a CTA may use (227 KB)

// Tile geometry.  WN weight rows per tile; the ring takes as many stages as fit in
// the shared memory beside the staging rows of a staged epilogue (STG), at most 8:
// with the lo token tile (LO), 256 -> 3 stages of 64 KB and 128 -> 4 of 48 KB;
// without it, 256 -> 4 of 48 KB and 128 -> 6 of 32 KB (7 without staging).
// CG = 2 (CTA pairs, WN = 256): each CTA holds one 128-row half of the weight tile,
// so a stage is 32 KB (48 KB with LO) and 6 or 7 (4) stages fit.
template <bool GU, int WN, bool LO, int CG = 1, bool STG = !GU> struct Geo {
    static_assert(WN == 128 || WN == 256, "weight tile width");
    static_assert(!GU || WN == 256, "gate/up tiles hold 128 gate + 128 up rows");
    static_assert(CG == 1 || WN == 256, "CTA pairs split a 256-row weight tile");
    static constexpr uint32_t TILE_W = WN / CG * BK * 2;             // this CTA's weight rows
    static constexpr uint32_t STAGE = TILE_W + (LO ? 2 : 1) * TILE_X;   // W, X hi[, X lo]
    static constexpr size_t EPI = STG ? EPI_BYTES : 0;
    static constexpr int FIT = (int)((SMEM_MAX - 1024 - 256 - EPI) / STAGE);
    static constexpr int STAGES = FIT < 8 ? FIT : 8;
    static constexpr uint32_t TMEM_COLS = 2 * WN;           // two tiles in flight
    static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE + EPI + 256;
};

// What a launch computes.  Dense: token rows [0, m_tok) in tiles of BT.  Grouped
// (tiles != nullptr): token tile j is (expert e, first grouped row r0) from the
// tile list, rows [r0, off[e+1]) of the grouped activations, and expert e's weight
// rows start at e * n_out.  Weight blocks: ceil(n_out / WN); for GU, n_out is the
// number of gate rows (= up rows) and a block is 128 features.
struct Args {
    int n_out;        // weight rows (per expert when grouped)
    int k;            // reduction length, a multiple of BK
    int x_col0;       // first activation column read (a multiple of 8)
    int piece_rows;   // dense: rows of map w0 before map w1 starts (0: w0 only); a multiple of 128
    int m_tok;        // token rows (grouped: the bound of the gathered source rows)
    int ksplit;       // dense, one CTA per tile: the reduction is cut into ksplit equal parts
                      // (0 or 1: none); part s of a tile reaches the functor as e = s
    const int *tiles; // grouped: [0] = count, then (expert, first row) pairs
    const int *off;   // grouped: expert row offsets [E + 1]
    int *status;      // DS4G_ETIMEOUT on a wait that gave up
    // gathering launches: grouped row r reads activation row grow[r] / gdiv of the
    // row-major BF16 arrays gx_hi, gx_lo (row stride gld elements)
    const int *grow;
    int gdiv;
    const bf16 *gx_hi, *gx_lo;
    int gld;
};

// An arrive-on of *bar that fires once every earlier cp.async of this thread has
// completed; the barrier's expected count includes this arrival (noinc).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

struct NoAux {};
template <class Epi, bool GU> struct AuxOf { using type = typename Epi::Aux; };
template <class Epi> struct AuxOf<Epi, true> { using type = NoAux; };   // gate/up: no functor loads
// Epilogue form of a (non gate/up) functor: Epi::kDirect selects the per-token form.
template <class Epi, bool GU> struct DirectOf { static constexpr bool value = Epi::kDirect; };
template <class Epi> struct DirectOf<Epi, true> { static constexpr bool value = false; };
template <class Epi, bool GU> __host__ __device__ constexpr bool staged_epi() { return !GU && !DirectOf<Epi, GU>::value; }

// A warp's staging rows: token t's 32 features as 8 float4 groups, group g stored at
// slot g ^ (t & 7), so that eight threads writing (or reading) the same group of
// eight tokens, or one token's eight groups, hit distinct banks.
__device__ __forceinline__ void stage_row(float *wstg, int t, const float (&v)[32])
{
    float4 *row = reinterpret_cast<float4 *>(wstg + t * CH);
#pragma unroll
    for (int g = 0; g < CH / 4; ++g) row[g ^ (t & 7)] = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
}
__device__ __forceinline__ float4 staged(const float *wstg, int t, int g)
{
    return reinterpret_cast<const float4 *>(wstg + t * CH)[g ^ (t & 7)];
}

// GU: the tile's gate rows come from w0 and its up rows from w1 (same row index);
// the epilogue calls Epi::store_row(m, i0, h[32], e) with h = silu(gate) * up of
// features i0 .. i0 + 31 of token m.  Otherwise, with Epi::kDirect, Epi provides
// Aux load32(m, f0, e) (what the features f0 .. f0 + 31 of token m need from global
// memory) and store32(m, f0, v[32], aux, e), called by the thread that owns token m;
// without it, Aux load4(m, n, e) and store4(m, n, v[4], aux, e) for four features,
// the chunk staged through shared memory so that an instruction covers 4 tokens x 32
// features (coalesced read-modify-write of the residual, for one).
// GA (grouped only): the token tiles are gathered row by row from a.gx_hi / a.gx_lo
// by GWARPS extra warps with 16-byte cp.async copies (the maps xhi, xlo are unused).
// LO: the activations' lo half takes part (two MMAs per K step); without it the
// products are taken with the BF16 activations alone (xlo / gx_lo are not read).
// CG = 2 (dense only; launched in clusters of 2): the two CTAs of a cluster compute
// the two token tiles 2j, 2j + 1 against the same 256 weight rows with one
// tcgen05.mma.cta_group::2 of M = 256 per K step, issued by the even CTA.  Each CTA
// loads its own token tile and one 128-row half of the weight tile (the even CTA
// the first half; for GU the gate rows, the odd one the up rows), both completing
// on the even CTA's full barrier; the MMA completions arrive on both CTAs' empty
// and accumulator barriers (multicast commit), and the epilogue warps of both
// report a drained accumulator to the even CTA.  Per CTA and K step the tensor core
// reads half the weight bytes from shared memory, and TMA writes half as many.
template <class Epi, bool GU, int WN, bool GA, bool LO, int CG = 1>
__global__ void __launch_bounds__(GA ? THREADS_GA : THREADS, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap w0, const __grid_constant__ CUtensorMap w1,
              const __grid_constant__ CUtensorMap xhi, const __grid_constant__ CUtensorMap xlo,
              const Args a, const Epi epi)
{
    static_assert(CG == 1 || (CG == 2 && !GA), "CTA pairs: dense GEMMs");
    constexpr bool STG = staged_epi<Epi, GU>();
    using G = Geo<GU, WN, LO, CG, STG>;
    constexpr int STAGES = G::STAGES;
    constexpr uint32_t STAGE_BYTES = G::STAGE;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float *stg = reinterpret_cast<float *>(sm + STAGES * STAGE_BYTES);   // epilogue staging (STG)
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + STAGES * STAGE_BYTES + G::EPI);
    uint64_t *empty = full + STAGES;
    uint64_t *accf = empty + STAGES;   // [2] accumulator ready (MMA commit)
    uint64_t *acce = accf + 2;         // [2] accumulator drained (256 epilogue threads; CG 2: 16 warps)
    uint64_t *done = acce + 2;         // every MMA of this CTA completed
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);
    int *abort_flag = reinterpret_cast<int *>(tslot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int mtiles = GU ? a.n_out / BOXW : (a.n_out + WN - 1) / WN;
    // Split reductions (CG 1, dense): ksplit work items per tile, one per part.
    const int ksplit = CG == 1 && !a.tiles && a.ksplit > 1 ? a.ksplit : 1;
    const int nk = a.k / ksplit / BK;
    const int rank = CG == 2 ? (int)cluster_rank() : 0;
    const bool leader = rank == 0;
    const int first = blockIdx.x / CG, stride = gridDim.x / CG;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // TMA, and each gather lane
            mbar_init(&full[s], GA ? 1 + 32 * GWARPS : 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], CG == 2 ? 16 : 256);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc<CG>(tslot, G::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync_all();   // the peer's barriers exist before any remote use
    tc_fence_after();
    // with a programmatic launch the set-up above overlaps the previous kernel's tail;
    // its outputs (this GEMM's inputs) are complete past this point
    pdl_wait();
    pdl_trigger();
    // The grouped tile list is an output of an earlier kernel: read only past pdl_wait.
    // CG 2: a work item is a pair of token tiles; the cluster's CTAs share it.
    const int ntiles = a.tiles ? a.tiles[0] : (a.m_tok + BT - 1) / BT;
    const int total = mtiles * (CG == 2 ? (ntiles + 1) / 2 : ntiles) * ksplit;
    // tile -> (weight block mb, expert e, first token row r0, end row)
    auto tile_of = [&](int tau, int &mb, int &e, int &r0, int &rend) {
        mb = tau % mtiles;
        const int j = tau / mtiles;
        if (CG == 2) {
            e = 0;
            r0 = (2 * j + rank) * BT;
            rend = min(r0 + BT, a.m_tok);   // <= r0: no token of this CTA in the tile
        } else if (a.tiles) {
            e = a.tiles[1 + 2 * j];
            r0 = a.tiles[2 + 2 * j];
            rend = min(r0 + BT, a.off[e + 1]);
        } else {
            e = j / ntiles;   // the part of a split reduction (0 without)
            r0 = (j % ntiles) * BT;
            rend = min(r0 + BT, a.m_tok);
        }
    };
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
            if (LO) tma_prefetch_desc(&xlo);
            unsigned it = 0;
            bool ok = true;
            constexpr int NB = WN / BOXW / CG;   // 128-row weight boxes this CTA loads
            for (int tau = first; ok && tau < total; tau += stride) {
                int mb, e, r0, rend;
                tile_of(tau, mb, e, r0, rend);
                const int we = a.tiles ? e : 0;   // the expert (grouped) whose weights are read
                const int ks = a.tiles ? 0 : e;   // the reduction part (dense; 0 unless split)
                // the tile's weight boxes: (map, first row) of each 128-row box
                const void *bm[NB];
                int brow[NB];
#pragma unroll
                for (int hb = 0; hb < NB; ++hb) {
                    const int h = hb + rank;   // CG 2: this CTA's half
                    if (GU) {
                        bm[hb] = h ? &w1 : &w0;
                        brow[hb] = we * a.n_out + mb * BOXW;
                    } else {
                        int row = mb * WN + h * BOXW;
                        if (row >= a.n_out) row = mb * WN;   // ragged last block: its features are skipped
                        if (a.piece_rows > 0 && row >= a.piece_rows) {
                            bm[hb] = &w1;
                            brow[hb] = row - a.piece_rows;
                        } else {
                            bm[hb] = &w0;
                            brow[hb] = we * a.n_out + row;
                        }
                    }
                }
                for (int i = 0; i < nk; ++i, ++it) {
                    const int s = it % STAGES;
                    if (!mbar_wait(&empty[s], ((it / STAGES) & 1) ^ 1, ab)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    unsigned char *st = sm + s * STAGE_BYTES;
                    const int kx = (ks * nk + i) * BK;
                    if constexpr (CG == 2) {
                        // both CTAs' copies complete on the even CTA's full barrier, whose
                        // one arrival expects the bytes of both (the odd CTA's copies may
                        // land first: the transaction count goes below zero meanwhile, and
                        // the phase cannot complete before the arrival)
                        const uint32_t fb = cluster_map(&full[s], 0);
                        if (leader) mbar_expect_tx(&full[s], 2 * STAGE_BYTES);
                        tma_load_2d_pair(st, bm[0], kx, brow[0], fb);
                        tma_load_2d_pair(st + G::TILE_W, &xhi, a.x_col0 + kx, r0, fb);
                        if constexpr (LO) tma_load_2d_pair(st + G::TILE_W + TILE_X, &xlo, a.x_col0 + kx, r0, fb);
                        continue;
                    }
                    mbar_expect_tx(&full[s], GA ? G::TILE_W : STAGE_BYTES);
#pragma unroll
                    for (int h = 0; h < NB; ++h) tma_load_2d(st + h * BOX_BYTES, bm[h], kx, brow[h], &full[s]);
                    if constexpr (!GA) {
                        tma_load_2d(st + G::TILE_W, &xhi, a.x_col0 + kx, r0, &full[s]);
                        if constexpr (LO) tma_load_2d(st + G::TILE_W + TILE_X, &xlo, a.x_col0 + kx, r0, &full[s]);
                    }
                }
            }
            // no copy may still be in flight when the CTA exits (CG 2: the copies complete
            // on the even CTA's barrier; the stage's release by the MMA implies them)
            const unsigned n = it < (unsigned)STAGES ? it : (unsigned)STAGES;
            for (unsigned q = 1; q <= n; ++q) {
                const unsigned i = it - q;
                volatile int never = 0;
                if constexpr (CG == 2)
                    mbar_wait(&empty[i % STAGES], (i / STAGES) & 1, &never);
                else
                    mbar_wait(&full[i % STAGES], (i / STAGES) & 1, &never);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && !leader) {
            // CG 2, odd CTA: the even CTA issues the pair's MMAs, which read this CTA's
            // shared memory and write its TMEM; wait for their completion
            volatile int never = 0;
            mbar_wait(done, 0, &never);
        } else if (lane == 0) {
            // ---------------- MMA issuer
            constexpr uint32_t idesc = idesc_bf16_f32(BT * CG, WN);
            unsigned it = 0, tc = 0;
            bool ok = true;
            for (int tau = first; ok && tau < total; tau += stride, ++tc) {
                const int b = tc & 1;
                if (!mbar_wait(&acce[b], ((tc >> 1) & 1) ^ 1, ab)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(b * WN);
                for (int i = 0; i < nk; ++i, ++it) {
                    const int s = it % STAGES;
                    if (!mbar_wait(&full[s], (it / STAGES) & 1, ab)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // gathered token rows were written by cp.async (generic proxy); the
                    // tensor core reads them through the async proxy
                    if constexpr (GA) fence_proxy_async_smem();
                    const uint32_t sa = smem_u32(sm + s * STAGE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t wd = sdesc_kmajor_sw128(sa + kk * 32);
                        const uint64_t xh = sdesc_kmajor_sw128(sa + G::TILE_W + kk * 32);
                        tc_mma_bf16<CG>(acc, xh, wd, idesc, (i | kk) != 0);
                        if constexpr (LO) {
                            const uint64_t xl = sdesc_kmajor_sw128(sa + G::TILE_W + TILE_X + kk * 32);
                            tc_mma_bf16<CG>(acc, xl, wd, idesc, 1u);
                        }
                    }
                    tc_commit<CG>(&empty[s]);   // the stage is free once these MMAs complete
                }
                if (ok) tc_commit<CG>(&accf[b]);   // the tile is complete once every MMA is
            }
            // TMEM may be freed only after every MMA issued here has completed
            tc_commit<CG>(done);
            volatile int never = 0;
            mbar_wait(done, 0, &never);
        }
    } else if (GA && warp >= THREADS / 32) {
        if constexpr (GA) {
            // ---------------- token-row gather (warps 10 ..): gather warp gw fills tile rows
            // [64 gw, 64 gw + 64), hi and lo, in the stage's 128-byte-swizzled token tiles
            // (16-byte chunk c of row t at chunk c ^ (t & 7) of its 128-byte row, as TMA lays
            // it).  Lane l copies chunk l % 8 of rows 4 q + l / 8, so that each copy
            // instruction reads four whole 128-byte row segments.  Every lane arrives on the
            // stage's full barrier through cp.async.mbarrier.arrive.noinc: the arrival fires
            // when the lane's copies have landed, so the warp never waits for its copies and
            // runs as far ahead as the free stages allow (the L2 latency of the token rows
            // under a saturated weight stream is longer than two stages).  Rows past the
            // group's end are not copied: their products only reach accumulator rows the
            // epilogue skips.
            const int gw = warp - THREADS / 32, c = lane & 7;
            unsigned it = 0;
            bool ok = true;
            for (int tau = first; ok && tau < total; tau += stride) {
                int mb, e, r0, rend;
                tile_of(tau, mb, e, r0, rend);
                int src[16];   // source row of this lane's tile rows in gx (-1: not copied)
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const int r = r0 + 64 * gw + 4 * q + (lane >> 3);
                    src[q] = -1;
                    if (r < rend) {
                        const int v = a.grow[r] / a.gdiv;
                        if ((unsigned)v < (unsigned)a.m_tok) src[q] = v;
                        else atomicCAS(a.status, 0, DS4G_EINVAL);   // not a token of this launch: never copied
                    }
                }
                const int col = a.x_col0 + 8 * c;
                for (int i = 0; i < nk; ++i, ++it) {
                    const int s = it % STAGES;
                    if (!mbar_wait(&empty[s], ((it / STAGES) & 1) ^ 1, ab)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    unsigned char *xt = sm + s * STAGE_BYTES + G::TILE_W;
                    const int kx = i * BK;
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        if (src[q] < 0) continue;
                        const int row = 64 * gw + 4 * q + (lane >> 3);
                        const int off = row * 128 + ((c ^ (row & 7)) << 4);
                        const size_t so = (size_t)src[q] * a.gld + col + kx;
                        cp_async16(xt + off, a.gx_hi + so);
                        if constexpr (LO) cp_async16(xt + TILE_X + off, a.gx_lo + so);
                    }
                    cp_async_arrive_noinc(&full[s]);
                }
            }
            cp_async_wait_all();   // nothing in flight at exit
        }
    } else {
        // ---------------- epilogue (warps 2-9): warp w reads TMEM lane quarter w % 4
        // (tokens 32q ..) and takes every other 32-feature chunk of the tile; each
        // thread owns one token (its TMEM lane) and hands the functor the chunk's 32
        // adjacent features of it, so RoPE pairs and 16-byte stores stay in registers
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        const int tok = 32 * q + lane;     // this thread's token row in the tile
        // the accumulator is drained: every thread (CG 1), or each warp to the even CTA (CG 2)
        auto drained = [&](int b) {
            tc_fence_before();
            if constexpr (CG == 2) {
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(cluster_map(&acce[b], 0));
            } else {
                mbar_arrive(&acce[b]);
            }
        };
        using Aux = typename AuxOf<Epi, GU>::type;
        // staged form: a batch of the functor's loads for chunk c, items (token, 4 features)
        auto load_batch = [&](const auto &ep, int mb, int e, int r0, int rend, int c, auto &ax) {
            const int f0 = mb * WN + c * CH;
#pragma unroll
            for (int u = 0; u < EPI_BATCH; ++u) {
                const int idx = lane + 32 * u;
                const int t = idx >> 3, j = (idx & 7) * 4, mm = r0 + 32 * q + t;
                if (mm < rend && f0 + j < a.n_out) ax[u] = ep.load4(mm, f0 + j, e);
            }
        };
        unsigned tc = 0;
        for (int tau = first; tau < total; tau += stride, ++tc) {
            int mb, e, r0, rend;
            tile_of(tau, mb, e, r0, rend);
            const int b = tc & 1;
            const bool wlive = r0 + 32 * q < rend;   // warp-uniform: any token of this warp in the tile
            const int m = r0 + tok;
            const bool tlive = m < rend;
            // The functor's loads depend on the tile's coordinates only: the first chunk's
            // are issued before the accumulator is ready, each later chunk's while the
            // previous chunk is stored.
            Aux aux[2];                       // direct form: per thread and chunk
            Aux sax[STG ? 2 : 1][EPI_BATCH];  // staged form: per item of a batch
            if constexpr (STG) {
                if (wlive) load_batch(epi, mb, e, r0, rend, half, sax[0]);
            } else if constexpr (!GU) {
                if (tlive && mb * WN + half * CH < a.n_out) aux[0] = epi.load32(m, mb * WN + half * CH, e);
            }
            if (!mbar_wait(&accf[b], (tc >> 1) & 1, ab)) {
                give_up();
                break;
            }
            tc_fence_after();
            const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * WN);
            if constexpr (GU) {
                // gate columns c, up columns 128 + c of this thread's token
#pragma unroll 1
                for (int c0 = 32 * half; c0 < BOXW; c0 += 64) {
                    float g[32], u[32];
                    if (wlive) {
                        tmem_ld32(lane_base + (uint32_t)c0, g);
                        tmem_ld32(lane_base + (uint32_t)(BOXW + c0), u);
                    }
                    if (c0 + 64 >= BOXW) drained(b);   // this warp's share of the accumulator
                    if (wlive && tlive) {
                        float h[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) h[j] = silu_mul(g[j], u[j]);
                        epi.store_row(m, mb * BOXW + c0, h, e);
                    }
                }
            } else if constexpr (!STG) {
                constexpr int NCW = WN / CH / 2;   // chunks per warp: half, half + 2, ...
#pragma unroll
                for (int k = 0; k < NCW; ++k) {
                    const int f0 = mb * WN + (half + 2 * k) * CH;
                    float v[32];
                    if (wlive) tmem_ld32(lane_base + (uint32_t)(f0 - mb * WN), v);
                    if (k == NCW - 1) drained(b);   // this warp's last chunk is read
                    if (!wlive || !tlive) continue;
                    if (k + 1 < NCW && f0 + 2 * CH < a.n_out) aux[(k + 1) & 1] = epi.load32(m, f0 + 2 * CH, e);
                    if (f0 < a.n_out) epi.store32(m, f0, v, aux[k & 1], e);
                }
            } else {
                // staged: the chunk goes through this warp's staging rows; an item is (token,
                // 4 features), an instruction covers 4 tokens x 32 features, and a chunk's
                // functor loads (eight per thread) are issued one chunk ahead
                float *wstg = stg + (warp - 2) * 32 * CH;   // this warp's [32 tokens][CH] rows
                constexpr int NCW = WN / CH / 2;
#pragma unroll
                for (int k = 0; k < NCW; ++k) {
                    const int c = half + 2 * k;
                    float v[32];
                    if (wlive) tmem_ld32(lane_base + (uint32_t)(c * CH), v);
                    if (k == NCW - 1) drained(b);
                    if (!wlive) continue;
                    stage_row(wstg, lane, v);
                    if (k + 1 < NCW) load_batch(epi, mb, e, r0, rend, c + 2, sax[(k + 1) & 1]);
                    __syncwarp();
                    const int f0 = mb * WN + c * CH;
#pragma unroll
                    for (int u = 0; u < EPI_BATCH; ++u) {
                        const int idx = lane + 32 * u;
                        const int t = idx >> 3, j = (idx & 7) * 4, mm = r0 + 32 * q + t;
                        if (mm >= rend || f0 + j >= a.n_out) continue;
                        const float4 v4 = staged(wstg, t, j >> 2);
                        const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
                        epi.store4(mm, f0 + j, vv, sax[k & 1][u], e);
                    }
                    __syncwarp();   // the staging rows are rewritten next
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    // CG 2: neither CTA leaves while the other may still signal its barriers
    if constexpr (CG == 2) cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem, G::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side

// Tensor map of a row-major BF16 matrix [rows][cols] (row stride ld elements) read
// in boxes of 64 columns x box_rows rows with the 128-byte swizzle; rows beyond
// `rows` read as zeros.
cudaError_t make_map_bf16(CUtensorMap *m, const void *base, int rows, int cols, int ld, int box_rows);

template <bool GU, int WN, bool LO, class Epi, bool GA = false>
static cudaError_t launch_wn(const CUtensorMap &w0, const CUtensorMap &w1, const CUtensorMap &xhi,
                             const CUtensorMap &xlo, const Args &a, const Epi &epi, long long work, int nsm,
                             cudaStream_t st)
{
    static bool attr_set = false;   // per instantiation; set before the first launch
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_tc_gemm<Epi, GU, WN, GA, LO>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)Geo<GU, WN, LO, 1, staged_epi<Epi, GU>()>::SMEM);
        if (e) return e;
        attr_set = true;
    }
    const int grid = (int)(work < nsm ? work : nsm);
    return launch_pdl(k_tc_gemm<Epi, GU, WN, GA, LO>, dim3(grid), dim3(GA ? THREADS_GA : THREADS),
                      Geo<GU, WN, LO, 1, staged_epi<Epi, GU>()>::SMEM, st, w0, w1, xhi, xlo, a, epi);
}

// The CTA-pair form (256-row weight tiles, dense): clusters of 2, as many as can be
// resident at once (some GPCs may hold an odd number of SMs), at most one per pair of
// token tiles and weight block.  0 clusters resident: cudaErrorNotSupported.
template <bool GU, bool LO, class Epi>
static cudaError_t launch_pair(const CUtensorMap &w0, const CUtensorMap &w1, const CUtensorMap &xhi,
                               const CUtensorMap &xlo, const Args &a, const Epi &epi, long long work,
                               cudaStream_t st)
{
    auto kern = k_tc_gemm<Epi, GU, 256, false, LO, 2>;
    constexpr size_t smem = Geo<GU, 256, LO, 2, staged_epi<Epi, GU>()>::SMEM;
    static int clusters = -1;   // per instantiation: resident clusters of 2
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    if (clusters < 0) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e) return e;
        cfg.gridDim = dim3(2);
        cfg.numAttrs = 1;
        int n = 0;
        if ((e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg))) return e;
        clusters = n;
    }
    if (clusters <= 0) return cudaErrorNotSupported;
    const long long nc = work < clusters ? work : clusters;
    cfg.gridDim = dim3((unsigned)(2 * nc));
    cfg.numAttrs = 2;
    ++launch_count();
    return cudaLaunchKernelEx(&cfg, kern, w0, w1, xhi, xlo, a, epi);
}

// ntile_bound: token tiles at most (dense: exact; grouped: the tile list's bound).
// Dense GEMMs whose 256-row weight blocks times token-tile pairs give every SM pair
// a work item run on CTA pairs; other plain GEMMs take 256-row weight tiles when
// that still gives every SM two tiles, else 128-row tiles (twice the tiles, half the
// reuse of each token tile).
template <bool GU, bool LO, class Epi>
static cudaError_t launch(const CUtensorMap &w0, const CUtensorMap &w1, const CUtensorMap &xhi,
                          const CUtensorMap &xlo, const Args &a, const Epi &epi, int ntile_bound, int nsm,
                          cudaStream_t st)
{
    if (ntile_bound <= 0 || a.n_out <= 0) return cudaSuccess;
    const long long blocks256 = GU ? a.n_out / BOXW : (a.n_out + 255) / 256;
    const long long parts = !a.tiles && a.ksplit > 1 ? a.ksplit : 1;
    if (!a.tiles && ntile_bound >= 2 && parts == 1) {
        const long long pairs = blocks256 * ((ntile_bound + 1) / 2);
        if (2 * pairs >= nsm) return launch_pair<GU, LO>(w0, w1, xhi, xlo, a, epi, pairs, st);
    }
    if constexpr (GU) {
        const long long work = blocks256 * ntile_bound;
        if (a.grow) return launch_wn<true, 256, LO, Epi, true>(w0, w1, xhi, xlo, a, epi, work, nsm, st);
        return launch_wn<true, 256, LO>(w0, w1, xhi, xlo, a, epi, work, nsm, st);
    } else {
        const long long w256 = blocks256 * ntile_bound * parts;
        if (w256 >= 2ll * nsm) return launch_wn<false, 256, LO>(w0, w1, xhi, xlo, a, epi, w256, nsm, st);
        return launch_wn<false, 128, LO>(w0, w1, xhi, xlo, a, epi,
                                         (long long)((a.n_out + 127) / 128) * ntile_bound * parts, nsm, st);
    }
}

}  // namespace tc
}  // namespace ds4g
