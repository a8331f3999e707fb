// Tensor-core form of the layer-major prefill (prefill_tc.cu): TMA tensor maps of
// one layer's weights and of a session's prefill activations, and the chunk pass.
#pragma once

#include <cuda.h>

#include "kernels.h"

namespace ds4g {

struct TcLayerMaps {   // boxes: 64 columns x 128 rows
    CUtensorMap wqa, wkva, wqb, wkb, wvb, wo, wr, wsg, wsu, wsd, wg, wu, wd;
};
struct TcActPtrs {     // hi/lo BF16 halves of the prefill activation buffers
    bf16 *xn_hi, *xn_lo, *c_hi, *c_lo, *o_hi, *o_lo, *hg_hi, *hg_lo, *hs_hi, *hs_lo;
};
struct TcActMaps {     // boxes: 64 columns x 128 token rows (q, oa: x 128 [token][head] rows)
    CUtensorMap xn_hi, xn_lo, c_hi, c_lo, o_hi, o_lo, hg_hi, hg_lo, hs_hi, hs_lo, q_hi, q_lo, oa_hi,
        oa_lo;
};
struct TcKVMaps {      // one layer's K and V cache, boxes: 64 dims x the attention's staged key rows
    CUtensorMap k, v;
};

// Shapes the tensor-core form covers: BF16 weights; every weight piece a multiple
// of 128 rows and every reduction a multiple of 64.
bool tc_prefill_eligible(const Dims &d);
// Tensor-core attention for the prefill (head dim 128, window <= 128, BF16 KV).
bool attn_mma_eligible(const Dims &d);
cudaError_t attn_mma_setup(const Dims &d, int max_smem);
// Tensor-core attention for the prefill on tcgen05 (attn_tc.cu): head dim 128, NH
// in {16, 32, 64, 128}, window <= 128, BF16 KV; queries as BF16 hi/lo.
bool attn_tc_eligible(const Dims &d);
size_t attn_tc_smem(const Dims &d);
cudaError_t attn_tc_setup(const Dims &d, int max_smem);
cudaError_t attn_tc_kv_maps(const Dims &d, const void *kc, const void *vc, int n_ctx, TcKVMaps &m);
// Map of a [P * NH][128] BF16 array of [token][head] rows in 128-row boxes.
cudaError_t attn_tc_row_map(const Dims &d, int P, const bf16 *base, CUtensorMap &m);
// hilo: queries, probabilities and output as BF16 hi/lo pairs; otherwise single BF16.
cudaError_t attn_prefill_tc(const Dims &d, const CUtensorMap &qhi, const CUtensorMap &qlo, const TcKVMaps &kv,
                            const CUtensorMap &ohi, const CUtensorMap &olo, int p0, int n, int *status,
                            cudaStream_t st, int nsm, bool hilo);
cudaError_t tc_layer_maps(const Dims &d, const LayerPtrs &w, TcLayerMaps &m);
TcActPtrs tc_act_ptrs(const Dims &d, const PrefillBufs &pb);
cudaError_t tc_act_maps(const Dims &d, const PrefillBufs &pb, TcActMaps &m);
// kvm: per-layer K/V maps for the tcgen05 attention (nullptr: the warp-MMA one).
// hilo: every GEMM takes its activations as BF16 hi/lo pairs; otherwise only the
// router's (the other GEMMs multiply BF16 activations).
cudaError_t prefill_chunk_tc(const Dims &d, const LayerPtrs *layers, const TcLayerMaps *lm,
                             const TcActMaps &am, const TcKVMaps *kvm, void *const *kc, void *const *vc,
                             const float2 *rope, const uint16_t *tok_embd, const PrefillBufs &pb, int p0, int n,
                             cudaStream_t st, int nsm, bool hilo);

// prefill.cu kernels the tensor-core form shares
__global__ void k_embed_rows(const uint16_t *table, const int *tok, float *X, int H);
__global__ void k_router_topk(const float *S, int nparts, size_t part, int *ids, float *wts, int n, int E, int K,
                              int *status);
template <typename TKV>
cudaError_t attn_prefill_hilo(const Dims &d, const float *Q, bf16 *o_hi, bf16 *o_lo, const TKV *kc,
                              const TKV *vc, int p0, int n, cudaStream_t st);

}  // namespace ds4g
