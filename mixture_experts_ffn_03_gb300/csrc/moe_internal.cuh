// Internal interfaces between the host driver (moe_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace moe {

// Device status word bits (workspace status block, word 0).
enum : unsigned {
    ERR_GATE_UP_TIMEOUT = 1u << 0,
    ERR_DOWN_TIMEOUT = 1u << 1,
};

// Status block layout (int32 words at the start of the workspace).
enum : int {
    META_ERR = 0,          // device error flags
    META_RT_GU = 1,        // routed row tiles of the gate_up GEMM
    META_RT_DN = 2,        // routed row tiles of the down GEMM
    META_TICKET = 3,       // block-completion counter of the count/scan kernel
    META_WORDS = 64,
};

constexpr int kRouteWarps = 8;          // tokens per route block (one warp each)
constexpr int kCountTokens = 256;       // tokens per histogram block
constexpr int kGemmBM = 128;            // weight rows (output features) per tile
constexpr int kGemmBK = 64;             // K elements per pipeline stage

// Routing, histogram/scan, scatter and combine (moe_route.cu).
cudaError_t launch_route(int T, int H, int E, int k, int score_fn, const float* logits,
                         const __nv_bfloat16* hidden, const __nv_bfloat16* w_g, int* topk_ids,
                         float* topk_w, float* gate_logit, int* ids_out, float* w_out, int* meta,
                         cudaStream_t st);
cudaError_t launch_count_scan(int T, int E, int k, int bn_gu, int bn_dn, const int* topk_ids,
                              int* blockhist, int* counts, int* offsets, int2* rt_gu,
                              int2* rt_dn, int* meta, int* counts_out, cudaStream_t st);
cudaError_t launch_scatter(int T, int E, int k, const int* topk_ids, const int* blockhist,
                           const int* offsets, int* perm, int* inv, cudaStream_t st);
cudaError_t launch_combine(int T, int H, int k, const float* y, const float* topk_w,
                           const int* inv, __nv_bfloat16* out, cudaStream_t st);

// Grouped GEMMs (moe_gemm.cu).
struct GemmArgs {
    int T, H, E, k, I, I_s;
    const __nv_bfloat16* hidden;
    const int* perm;
    const int* counts;
    const int* offsets;
    const int2* rowtiles;   // routed row tiles (expert, first row) of this GEMM
    const int* meta;
    const float* gate_logit;
    __nv_bfloat16* h_hi;
    __nv_bfloat16* h_lo;
    __nv_bfloat16* hs_hi;
    __nv_bfloat16* hs_lo;
    float* y;
    unsigned* err;
};

struct GemmMaps {
    CUtensorMap w;      // gate_up: W_gate_up as [E*2I, H]; down: W_down as [E*H, I]
    CUtensorMap ws;     // gate_up: Ws_gate_up [2I_s, H]; down: Ws_down [H, I_s]
    CUtensorMap h_hi;   // down only: h_hi [T*k, I]
    CUtensorMap h_lo;
    CUtensorMap hs_hi;  // down only: hs_hi [T, I_s]
    CUtensorMap hs_lo;
};

// Supported tile widths (tokens per tile) of both GEMMs.
bool gemm_bn_supported(int bn);
cudaError_t launch_gate_up(int bn, const GemmMaps& maps, const GemmArgs& a, int max_tiles,
                           int num_sms, cudaStream_t st);
cudaError_t launch_down(int bn, const GemmMaps& maps, const GemmArgs& a, int max_tiles,
                        int num_sms, cudaStream_t st);

}  // namespace moe
