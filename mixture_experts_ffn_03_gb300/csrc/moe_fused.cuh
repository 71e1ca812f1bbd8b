// The fused expert phase (moe_fused.cu): gate_up and down of the bf16
// grouped GEMMs in one persistent launch, for batches whose gate_up and down
// tiles have the same width (at most 64 tokens).
#pragma once

#include "moe_internal.cuh"

namespace moe {

// Widest token tile the fused launch takes.
constexpr int kFusedMaxBN = 64;

// ready: one int per routed row tile (indexed by its first sorted row, 0 ..
// T*k-1) and per shared-expert row tile (T*k + its first token), zero at
// launch. a.rowtiles / a.sched are the gate_up GEMM's (both GEMMs use the
// same row tiles when their widths agree). max_tiles bounds the gate_up plus
// the down tiles.
cudaError_t launch_expert_fused(int bn, const GemmMaps& gu, const GemmMaps& dn, const GemmArgs& a,
                                int* ready, int max_tiles, int num_sms, cudaStream_t st);

// The whole layer in one launch (decode-sized batches: T*k <= kSmallSlots,
// E <= kLayerMaxExperts, equal tile widths of at most kFusedMaxBN): routing
// and the permute, the fused expert phase, the combine. What the separate
// routing and combine kernels take besides GemmArgs (whose gate_logit the
// routing writes here).
constexpr int kLayerMaxExperts = 256;
struct LayerArgs {
    int score_fn, bn_gu, bn_dn;
    LogitSrc logits;
    const __nv_bfloat16* w_g;
    int* topk_ids;
    float* topk_w;
    float* gate_logit;
    int* counts;
    int* offsets;
    int* perm;
    int* inv;
    int4* rt_gu;
    int4* rt_dn;
    int* meta;
    int* ids_out;
    float* w_out;
    int* counts_out;
    __nv_bfloat16* out;
};
cudaError_t launch_layer_fused(int bn, const GemmMaps& gu, const GemmMaps& dn, const GemmArgs& a,
                               int* ready, const LayerArgs& l, int num_sms, cudaStream_t st);

}  // namespace moe
