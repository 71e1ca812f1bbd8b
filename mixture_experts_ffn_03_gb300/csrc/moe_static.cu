// Allocation-free per-expert histogram: the counting step of the permute,
// with its scratch (per-block histograms and a completion ticket) in a
// file-scope device array instead of a caller-provided workspace.
//
// Who needs this: code that must not allocate device memory at all, such as
// a plugin behind a fixed interface that hands over only inputs and outputs
// and has no place to keep a workspace, or a latency-critical caller whose
// memory is fully pre-reserved and for which cudaMalloc (which can
// synchronise the device) is not allowed. This entry point performs no
// cudaMalloc/cudaFree and calls no allocating library routine.
//
// The array is part of the loaded library image: every GPU that loads the
// library holds it (1 MiB + 256 bytes) until the process exits. All calls
// share it, so calls that overlap on the GPU (different streams, or the same
// scratch used from several host threads without ordering) race on it.
#include "moe.h"
#include "moe_internal.cuh"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {
namespace {

constexpr int kTicketWords = 64;  // word 0: completion ticket; rest padding
static __device__ __align__(256) int g_static_scratch[kTicketWords + MOE_STATIC_HIST_WORDS];

// Device address of g_static_scratch in the current device's context. Host
// code must not use the symbol's name as an address. The address is looked
// up on every call (a cheap runtime query) rather than cached, so it stays
// right after the context is destroyed and recreated (cudaDeviceReset).
cudaError_t scratch_address(int** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    *out = static_cast<int*>(p);
    return cudaSuccess;
}

__global__ void __launch_bounds__(256)
expert_counts_static_kernel(int T, int E, int k, const int* __restrict__ topk_ids,
                            int* __restrict__ scratch, int* __restrict__ counts_out,
                            int* __restrict__ offsets_out) {
    extern __shared__ int s_hist[];  // [E]
    __shared__ int s_warp[8];
    __shared__ int s_is_last;
    int* ticket = scratch;
    int* blockhist = scratch + kTicketWords;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int e = tid; e < E; e += 256) s_hist[e] = 0;
    __syncthreads();
    const long a0 = static_cast<long>(blockIdx.x) * kCountTokens * k;
    const long a1 = min(static_cast<long>(T) * k, a0 + static_cast<long>(kCountTokens) * k);
    for (long a = a0 + tid; a < a1; a += 256) {
        const int e = topk_ids[a];
        if (e >= 0 && e < E) atomicAdd(&s_hist[e], 1);  // out-of-range ids are not counted
    }
    __syncthreads();
    for (int e = tid; e < E; e += 256) blockhist[static_cast<size_t>(blockIdx.x) * E + e] = s_hist[e];
    __threadfence();
    __syncthreads();
    if (tid == 0) s_is_last = (atomicAdd(ticket, 1) == static_cast<int>(gridDim.x) - 1);
    __syncthreads();
    if (!s_is_last) return;
    __threadfence();

    // Last block: totals per expert (thread tid owns experts tid*ept ..), then
    // an exclusive scan over experts in thread order.
    const int ept = (E + 255) / 256;
    int local[4] = {0, 0, 0, 0};
    int mine = 0;
    for (int r = 0; r < ept; ++r) {
        const int e = tid * ept + r;
        if (e >= E) break;
        int c = 0;
        for (int b = 0; b < static_cast<int>(gridDim.x); ++b)
            c += __ldcg(&blockhist[static_cast<size_t>(b) * E + e]);
        local[r] = c;
        mine += c;
    }
    int incl = mine;
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int run = incl - mine, total = 0;
    for (int w = 0; w < 8; ++w) {
        if (w < warp) run += s_warp[w];
        total += s_warp[w];
    }
    for (int r = 0; r < ept; ++r) {
        const int e = tid * ept + r;
        if (e >= E) break;
        counts_out[e] = local[r];
        if (offsets_out) offsets_out[e] = run;
        run += local[r];
    }
    if (tid == 0) {
        if (offsets_out) offsets_out[E] = total;
        *ticket = 0;
    }
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API moe_status moe_expert_counts_static(const int32_t* topk_ids, int32_t T, int32_t k,
                                            int32_t E, int32_t* counts_out,
                                            int32_t* offsets_out, void* cuda_stream) {
    if (T < 0 || k < 1 || k > 32 || E < 1 || E > 1024 || k > E || !counts_out)
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && !topk_ids) return MOE_ERR_INVALID_ARG;
    const long blocks = (static_cast<long>(T) + kCountTokens - 1) / kCountTokens;
    if (blocks * E > MOE_STATIC_HIST_WORDS) return MOE_ERR_CAPACITY;
    int* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    if (T == 0) {
        // No tokens: every count and offset is zero.
        if (cudaMemsetAsync(counts_out, 0, sizeof(int32_t) * E, st) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (offsets_out &&
            cudaMemsetAsync(offsets_out, 0, sizeof(int32_t) * (E + 1), st) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    // The completion ticket must start at zero; the previous call's last block
    // reset it, but a call that never ran to completion would not have.
    if (cudaMemsetAsync(scratch, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
    expert_counts_static_kernel<<<static_cast<int>(blocks), 256, E * sizeof(int), st>>>(
        T, E, k, topk_ids, scratch, counts_out, offsets_out);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
