// Routing, per-expert token lists and the final combine.
//
//   route       one warp per token: score, top-k (ties to the lower expert
//               index), renormalisation, and the shared-expert gate logit
//               x . w_g. Router in fp32, softmax or sigmoid score, normalised
//               top-k affinities: "Add Qwen3.5-35B-A3B (support vision and
//               text input)", Model Information and Additional Information.
//   count_scan  per-block expert histograms; the last block to finish turns
//               them into counts, exclusive offsets and the row-tile lists of
//               both grouped GEMMs.
//   scatter     stable scatter of (token, slot) pairs into expert-sorted
//               order: tokens ascending within each expert.
//   combine     out_t = bf16( sum_j w_tj y[inv(t,j)] + y_shared[t] ), summed
//               in fp32 in slot order, one rounding; gather-based, no atomics.
//               The expert output of "[RFC] Experimental Qwen3.5 MoE AFD
//               support: CUDA correctness baseline", Proposed plugin boundary.
#include "moe_internal.cuh"

namespace moe {
namespace {

// Order-preserving key of an fp32 logit: a larger key ranks first. -0 and +0
// are equal, NaN ranks below everything, so every bit pattern is placed.
__device__ __forceinline__ uint32_t rank_key(float v) {
    uint32_t b = __float_as_uint(v);
    if ((b & 0x7FFFFFFFu) == 0u) b = 0u;
    if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// One 64-bit code per (logit, expert): larger code ranks first; for equal
// logits the lower expert index has the larger code. Codes are distinct.
__device__ __forceinline__ uint64_t rank_code(float v, int e) {
    return (static_cast<uint64_t>(rank_key(v)) << 32) |
           static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(e));
}

__global__ void __launch_bounds__(kRouteWarps * 32)
route_kernel(int T, int H, int E, int k, int score_fn, const float* __restrict__ logits,
             const __nv_bfloat16* __restrict__ hidden, const __nv_bfloat16* __restrict__ w_g,
             int* __restrict__ topk_ids, float* __restrict__ topk_w,
             float* __restrict__ gate_logit, int* __restrict__ ids_out,
             float* __restrict__ w_out, int* __restrict__ meta) {
    extern __shared__ float s_rows[];  // [kRouteWarps][E]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        meta[META_ERR] = 0;
        meta[META_TICKET] = 0;
    }
    const int t = blockIdx.x * kRouteWarps + warp;
    if (t >= T) return;
    float* row = s_rows + warp * E;
    const float* lg = logits + static_cast<size_t>(t) * E;
    for (int e = lane; e < E; e += 32) row[e] = lg[e];
    __syncwarp();

    // Top-k: round j takes the best code strictly below the previous pick.
    uint64_t prev = ~0ull;
    float my_v = 0.f;
    int my_e = 0;
    for (int j = 0; j < k; ++j) {
        uint64_t best = 0;
        for (int e = lane; e < E; e += 32) {
            const uint64_t c = rank_code(row[e], e);
            if (c < prev && c > best) best = c;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
            best = other > best ? other : best;
        }
        prev = best;
        const int e_sel = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(best));
        if (lane == j) {
            my_e = e_sel;
            my_v = row[e_sel];
        }
    }

    // Renormalised scores of the selected experts. For softmax the full
    // partition function cancels in the renormalisation, leaving a softmax
    // over the selected logits (shifted by the largest one).
    float s;
    if (score_fn == 0) {
        const float m = __shfl_sync(0xFFFFFFFFu, my_v, 0);
        s = (lane < k) ? expf(my_v - m) : 0.f;
    } else {
        s = (lane < k) ? 1.f / (1.f + expf(-my_v)) : 0.f;
    }
    float sum = s;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (lane < k) {
        const float w = s / sum;
        const size_t o = static_cast<size_t>(t) * k + lane;
        topk_ids[o] = my_e;
        topk_w[o] = w;
        if (ids_out) ids_out[o] = my_e;
        if (w_out) w_out[o] = w;
    }

    // Shared-expert gate logit z_t = x_t . w_g, fp32 accumulation.
    const uint4* xr = reinterpret_cast<const uint4*>(hidden + static_cast<size_t>(t) * H);
    const uint4* gr = reinterpret_cast<const uint4*>(w_g);
    float acc = 0.f;
    for (int c = lane; c < H / 8; c += 32) {
        const uint4 a = xr[c], b = gr[c];
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 fa = __bfloat1622float2(a2[q]);
            const float2 fb = __bfloat1622float2(b2[q]);
            acc = fmaf(fa.x, fb.x, acc);
            acc = fmaf(fa.y, fb.y, acc);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) gate_logit[t] = acc;
}

// Exclusive scan of one int per thread over a 256-thread block.
__device__ int block_excl_scan_256(int v, int* s_warp, int* total) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    __syncthreads();
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const int x = s_warp[w];
        if (w < warp) base += x;
        tot += x;
    }
    *total = tot;
    return base + incl - v;
}

__global__ void __launch_bounds__(256)
count_scan_kernel(int T, int E, int k, int bn_gu, int bn_dn, const int* __restrict__ topk_ids,
                  int* __restrict__ blockhist, int* __restrict__ counts,
                  int* __restrict__ offsets, int2* __restrict__ rt_gu, int2* __restrict__ rt_dn,
                  int* __restrict__ meta, int* __restrict__ counts_out) {
    extern __shared__ int s_hist[];  // [E]
    __shared__ int s_warp[8];
    __shared__ int s_is_last;
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += 256) s_hist[e] = 0;
    __syncthreads();
    const long a0 = static_cast<long>(blockIdx.x) * kCountTokens * k;
    const long a1 = min(static_cast<long>(T) * k, a0 + static_cast<long>(kCountTokens) * k);
    for (long a = a0 + tid; a < a1; a += 256) atomicAdd(&s_hist[topk_ids[a]], 1);
    __syncthreads();
    for (int e = tid; e < E; e += 256) blockhist[static_cast<size_t>(blockIdx.x) * E + e] = s_hist[e];
    __threadfence();
    __syncthreads();
    if (tid == 0) s_is_last = (atomicAdd(&meta[META_TICKET], 1) == static_cast<int>(gridDim.x) - 1);
    __syncthreads();
    if (!s_is_last) return;
    __threadfence();

    // Last block: every histogram is visible. Thread tid owns the experts
    // [tid*ept, tid*ept + ept), so expert order is thread order.
    const int nb = gridDim.x;
    const int ept = (E + 255) / 256;  // <= 4 for E <= 1024
    int local[4] = {0, 0, 0, 0};
    int mine = 0;
    for (int r = 0; r < ept; ++r) {
        const int e = tid * ept + r;
        if (e >= E) break;
        int c = 0;
        for (int b = 0; b < nb; ++b) {
            int* p = &blockhist[static_cast<size_t>(b) * E + e];
            const int v = __ldcg(p);
            *p = c;  // becomes the block's base inside expert e
            c += v;
        }
        local[r] = c;
        mine += c;
    }
    int total;
    int run = block_excl_scan_256(mine, s_warp, &total);
    for (int r = 0; r < ept; ++r) {
        const int e = tid * ept + r;
        if (e >= E) break;
        counts[e] = local[r];
        offsets[e] = run;
        if (counts_out) counts_out[e] = local[r];
        run += local[r];
    }
    if (tid == 0) offsets[E] = total;

    // Row tiles (expert, first row) of both GEMMs; empty experts give none.
    for (int g = 0; g < 2; ++g) {
        const int bn = g == 0 ? bn_gu : bn_dn;
        int2* rt = g == 0 ? rt_gu : rt_dn;
        int nt = 0;
        for (int r = 0; r < ept; ++r) nt += (local[r] + bn - 1) / bn;
        int tot_tiles;
        int pos = block_excl_scan_256(nt, s_warp, &tot_tiles);
        for (int r = 0; r < ept; ++r) {
            const int e = tid * ept + r;
            if (e >= E) break;
            for (int m0 = 0; m0 < local[r]; m0 += bn) rt[pos++] = make_int2(e, m0);
        }
        if (tid == 0) meta[g == 0 ? META_RT_GU : META_RT_DN] = tot_tiles;
    }
    if (tid == 0) meta[META_TICKET] = 0;
}

__global__ void __launch_bounds__(256)
scatter_kernel(int T, int E, int k, const int* __restrict__ topk_ids,
               const int* __restrict__ blockhist, const int* __restrict__ offsets,
               int* __restrict__ perm, int* __restrict__ inv) {
    extern __shared__ int s_sub[];  // [8][E]: per-warp counts, then per-warp bases
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < 8 * E; i += 256) s_sub[i] = 0;
    __syncthreads();
    const long t0 = static_cast<long>(blockIdx.x) * kCountTokens + warp * 32;
    const long t1 = min(static_cast<long>(T), t0 + 32);
    const long wa0 = t0 * k, wa1 = t1 > t0 ? t1 * k : wa0;
    int* running = s_sub + warp * E;
    for (long a = wa0 + lane; a < wa1; a += 32) atomicAdd(&running[topk_ids[a]], 1);
    __syncthreads();
    for (int e = tid; e < E; e += 256) {
        int run = offsets[e] + blockhist[static_cast<size_t>(blockIdx.x) * E + e];
        for (int w = 0; w < 8; ++w) {
            const int v = s_sub[w * E + e];
            s_sub[w * E + e] = run;
            run += v;
        }
    }
    __syncthreads();
    // Ordered pass: chunks of 32 consecutive slots; equal experts inside a
    // chunk are ranked by lane, so slot order (token order) is kept.
    for (long base = wa0; base < wa1; base += 32) {
        const long a = base + lane;
        const int e = a < wa1 ? topk_ids[a] : -1;
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        int pos = 0;
        if (e >= 0) pos = running[e] + rank;
        __syncwarp();
        if (e >= 0 && (peers >> lane) == 1u) running[e] += __popc(peers);
        __syncwarp();
        if (e >= 0) {
            perm[pos] = static_cast<int>(a);
            inv[a] = pos;
        }
    }
}

__global__ void __launch_bounds__(256)
combine_kernel(int T, int H, int k, const float* __restrict__ y, const float* __restrict__ topk_w,
               const int* __restrict__ inv, __nv_bfloat16* __restrict__ out) {
    const int t = blockIdx.x;
    const int h = (blockIdx.y * 256 + threadIdx.x) * 4;
    if (h >= H) return;
    const size_t tk = static_cast<size_t>(t) * k;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int j = 0; j < k; ++j) {
        const float w = topk_w[tk + j];
        const int p = inv[tk + j];
        const float4 v = __ldcs(reinterpret_cast<const float4*>(y + static_cast<size_t>(p) * H + h));
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
    }
    const size_t srow = static_cast<size_t>(T) * k + t;
    const float4 s = __ldcs(reinterpret_cast<const float4*>(y + srow * H + h));
    acc.x += s.x;
    acc.y += s.y;
    acc.z += s.z;
    acc.w += s.w;
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&lo);
    packed.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(out + static_cast<size_t>(t) * H + h) = packed;
}

}  // namespace

cudaError_t launch_route(int T, int H, int E, int k, int score_fn, const float* logits,
                         const __nv_bfloat16* hidden, const __nv_bfloat16* w_g, int* topk_ids,
                         float* topk_w, float* gate_logit, int* ids_out, float* w_out, int* meta,
                         cudaStream_t st) {
    const int blocks = (T + kRouteWarps - 1) / kRouteWarps;
    const size_t smem = static_cast<size_t>(kRouteWarps) * E * sizeof(float);
    route_kernel<<<blocks, kRouteWarps * 32, smem, st>>>(T, H, E, k, score_fn, logits, hidden,
                                                          w_g, topk_ids, topk_w, gate_logit,
                                                          ids_out, w_out, meta);
    return cudaGetLastError();
}

cudaError_t launch_count_scan(int T, int E, int k, int bn_gu, int bn_dn, const int* topk_ids,
                              int* blockhist, int* counts, int* offsets, int2* rt_gu,
                              int2* rt_dn, int* meta, int* counts_out, cudaStream_t st) {
    const int blocks = (T + kCountTokens - 1) / kCountTokens;
    count_scan_kernel<<<blocks, 256, E * sizeof(int), st>>>(T, E, k, bn_gu, bn_dn, topk_ids,
                                                            blockhist, counts, offsets, rt_gu,
                                                            rt_dn, meta, counts_out);
    return cudaGetLastError();
}

cudaError_t launch_scatter(int T, int E, int k, const int* topk_ids, const int* blockhist,
                           const int* offsets, int* perm, int* inv, cudaStream_t st) {
    const int blocks = (T + kCountTokens - 1) / kCountTokens;
    scatter_kernel<<<blocks, 256, 8 * E * sizeof(int), st>>>(T, E, k, topk_ids, blockhist,
                                                             offsets, perm, inv);
    return cudaGetLastError();
}

cudaError_t launch_combine(int T, int H, int k, const float* y, const float* topk_w,
                           const int* inv, __nv_bfloat16* out, cudaStream_t st) {
    dim3 grid(T, (H / 4 + 255) / 256);
    combine_kernel<<<grid, 256, 0, st>>>(T, H, k, y, topk_w, inv, out);
    return cudaGetLastError();
}

}  // namespace moe
