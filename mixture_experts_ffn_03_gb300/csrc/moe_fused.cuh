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

}  // namespace moe
