// Routing, per-expert token lists and the final combine (the routing and
// small-batch permute device code is in routing.cuh).
//
//   combine     out_t = bf16( sum_j w_tj y[inv(t,j)] + y_shared[t] ), summed
//               in fp32 in slot order, one rounding; gather-based, no atomics.
//               The expert output of "[RFC] Experimental Qwen3.5 MoE AFD
//               support: CUDA correctness baseline", Proposed plugin boundary.
//
// Routing runs one warp per token. Batches with T*k <= kSmallSlots then
// permute inside the same launch: the last CTA to finish routing (a completion
// ticket) builds the whole sorted order (route_permute_kernel). Larger batches
// take two launches: route_count_kernel (routing plus per-block expert
// histograms; the last CTA scans them) and scatter_kernel, whose extra CTAs
// compute the shared-expert gate logits (they need nothing from routing, so
// they run beside the histogram scan instead of lengthening every routing
// warp).
#include "routing.cuh"

namespace moe {
namespace {

// ------------------------------------------------------------ small batches
// Routing of one token per CTA (warp 0 selects the experts; all eight warps
// share the gate logit's dot product, so the hidden row arrives in one round
// trip) plus, in the last CTA to finish, the complete permute of all
// T*k <= kSmallSlots slots.
template <int EPL>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_permute_kernel(int T, int H, int E, int k, int score_fn, int bn_gu, int bn_dn,
                     const LogitSrc logits, const __nv_bfloat16* __restrict__ hidden,
                     const __nv_bfloat16* __restrict__ w_g, int* __restrict__ topk_ids,
                     float* __restrict__ topk_w, float* __restrict__ gate_logit,
                     int* __restrict__ counts, int* __restrict__ offsets, int* __restrict__ perm,
                     int* __restrict__ inv, int4* __restrict__ rt_gu, int4* __restrict__ rt_dn,
                     int* __restrict__ meta, int* __restrict__ ids_out, float* __restrict__ w_out,
                     int* __restrict__ counts_out) {
    extern __shared__ int s_dyn[];
    __shared__ int s_warp[kRouteWarps];
    __shared__ float s_gate[kRouteWarps];
    __shared__ int s_is_last;
    const int tid = threadIdx.x;
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();  // no-op unless launched behind the router GEMM
    route_token_cta<EPL>(blockIdx.x, H, E, k, score_fn, logits, hidden, w_g, topk_ids, topk_w,
                         gate_logit, ids_out, w_out, s_gate);
    __threadfence();
    __syncthreads();
    if (tid == 0) s_is_last = (atomicAdd(&meta[META_TICKET], 1) == static_cast<int>(gridDim.x) - 1);
    __syncthreads();
    if (!s_is_last) return;
    __threadfence();
    permute_small(T, E, k, bn_gu, bn_dn, topk_ids, counts, offsets, perm, inv, rt_gu, rt_dn, meta,
                  counts_out, s_dyn, s_warp);
    if (tid == 0) meta[META_TICKET] = 0;
}

// ------------------------------------------------------------ large batches
// Last CTA of the large-batch routing launch: every block histogram
// blockhist[b][e] (slots of expert e among tokens [256 b, 256 b + 256)) is
// complete. Thread tid owns the experts [tid*ept, tid*ept + ept), so expert
// order is thread order: counts, exclusive offsets, both GEMMs' row tiles,
// and each block's base inside each expert (written over its histogram).
// Called by all 256 threads of the CTA; s_off and s_tstart are shared
// arrays of E + 1 ints.
__device__ __forceinline__ void scan_block_hist(int nb, int E, int bn_gu, int bn_dn,
                                                int* __restrict__ blockhist,
                                                int* __restrict__ counts,
                                                int* __restrict__ offsets, int4* __restrict__ rt_gu,
                                                int4* __restrict__ rt_dn, int* __restrict__ meta,
                                                int* __restrict__ counts_out, int* s_warp,
                                                int* s_off, int* s_tstart) {
    const int tid = threadIdx.x;
    const int ept = (E + 255) / 256;  // <= 4 for E <= 1024
    int local[4] = {0, 0, 0, 0};
    int mine = 0;
    for (int r = 0; r < ept; ++r) {
        const int e = tid * ept + r;
        if (e >= E) break;
        int c = 0;
        // 16 blocks' counts per round trip: all loads first, then the running
        // sum replaces each count by the block's base inside expert e.
        for (int b0 = 0; b0 < nb; b0 += 16) {
            int v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                v[j] = b0 + j < nb ? __ldcg(&blockhist[static_cast<size_t>(b0 + j) * E + e]) : 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (b0 + j < nb) blockhist[static_cast<size_t>(b0 + j) * E + e] = c;
                c += v[j];
            }
        }
        local[r] = c;
        mine += c;
    }
    int total;
    int run = block_excl_scan<8>(mine, s_warp, &total);
    const int first_off = run;
    for (int r = 0; r < ept; ++r) {
        const int e = tid * ept + r;
        if (e >= E) break;
        counts[e] = local[r];
        offsets[e] = run;
        if (counts_out) counts_out[e] = local[r];
        run += local[r];
    }
    if (tid == 0) offsets[E] = total;

    // Row tiles, written by all threads: a hot expert (thousands of tokens)
    // owns many tiles, which one thread would write one by one. s_off holds
    // the offsets, s_tstart each expert's first tile index.
    for (int r = 0, off = first_off; r < ept; ++r) {
        const int e = tid * ept + r;
        if (e >= E) break;
        s_off[e] = off;
        off += local[r];
    }
    if (tid == 0) s_off[E] = total;
    for (int g = 0; g < 2; ++g) {
        const int bn = g == 0 ? bn_gu : bn_dn;
        int nt = 0;
        for (int r = 0; r < ept; ++r) nt += (local[r] + bn - 1) / bn;
        int tot_tiles;
        int pos = block_excl_scan<8>(nt, s_warp, &tot_tiles);
        for (int r = 0; r < ept; ++r) {
            const int e = tid * ept + r;
            if (e >= E) break;
            s_tstart[e] = pos;
            pos += (local[r] + bn - 1) / bn;
        }
        if (tid == 0) s_tstart[E] = tot_tiles;
        __syncthreads();
        int4* rt = g == 0 ? rt_gu : rt_dn;
        for (int i = tid; i < tot_tiles; i += blockDim.x) {
            // the expert of tile i: the largest e with s_tstart[e] <= i (experts
            // without tiles share their start with the next expert that has some)
            int lo = 0, hi = E - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_tstart[mid] <= i) lo = mid;
                else hi = mid - 1;
            }
            const int m0 = (i - s_tstart[lo]) * bn;
            const int n_e = s_off[lo + 1] - s_off[lo];
            rt[i] = make_int4(lo, m0, min(bn, n_e - m0), s_off[lo] + m0);
        }
        if (tid == 0) meta[g == 0 ? META_RT_GU : META_RT_DN] = tot_tiles;
        __syncthreads();  // s_tstart is rewritten for the next GEMM
    }
}

// Routing of one token per warp plus the per-expert histogram of each block
// of 256 tokens, accumulated with integer atomics (the sums do not depend on
// their order) into blockhist, which starts at zero. The last CTA to finish
// (a completion ticket) scans the histograms: counts, offsets, row tiles and
// per-block bases for scatter_kernel. The gate logits are left to
// scatter_kernel.
// At most 64 registers: four CTAs per SM, so a 4096-token batch routes in
// one wave.
template <int EPL>
__global__ void __launch_bounds__(kRouteWarps * 32, 4)
route_count_kernel(int T, int E, int k, int score_fn, int bn_gu, int bn_dn,
                   const LogitSrc logits, int* __restrict__ topk_ids,
                   float* __restrict__ topk_w,
                   int* __restrict__ blockhist, int* __restrict__ counts,
                   int* __restrict__ offsets, int4* __restrict__ rt_gu, int4* __restrict__ rt_dn,
                   int* __restrict__ meta, int* __restrict__ ids_out, float* __restrict__ w_out,
                   int* __restrict__ counts_out) {
    __shared__ int s_warp[kRouteWarps];
    __shared__ int s_is_last;
    __shared__ int s_off[kMaxExperts + 1];
    __shared__ int s_tstart[kMaxExperts + 1];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();  // no-op unless launched behind the router GEMM
    const int t = blockIdx.x * kRouteWarps + warp;
    if (t < T) {
        const int e = route_and_store<EPL, false>(t, 0, E, k, score_fn, logits, nullptr, nullptr,
                                                  topk_ids, topk_w, nullptr, ids_out, w_out, lane);
        if (lane < k) atomicAdd(&blockhist[static_cast<size_t>(t / kCountTokens) * E + e], 1);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_is_last = (atomicAdd(&meta[META_TICKET], 1) == static_cast<int>(gridDim.x) - 1);
    __syncthreads();
    if (!s_is_last) return;
    __threadfence();
    const int nb = (T + kCountTokens - 1) / kCountTokens;
    scan_block_hist(nb, E, bn_gu, bn_dn, blockhist, counts, offsets, rt_gu, rt_dn, meta,
                    counts_out, s_warp, s_off, s_tstart);
    if (tid == 0) meta[META_TICKET] = 0;
}

// CTAs [0, ceil(T / 256)): the stable scatter of the slots of 256 tokens.
// CTAs from ceil(T / 256) on: the shared-expert gate logit z_t = x_t . w_g of
// eight tokens each, one warp per token (GateLogit's order). Those read only
// the layer's inputs and skip the wait for the routing launch.
__global__ void __launch_bounds__(256)
scatter_kernel(int T, int H, int E, int k, const int* __restrict__ topk_ids,
               const int* __restrict__ blockhist, const int* __restrict__ offsets,
               int* __restrict__ perm, int* __restrict__ inv,
               const __nv_bfloat16* __restrict__ hidden, const __nv_bfloat16* __restrict__ w_g,
               float* __restrict__ gate_logit) {
    extern __shared__ int s_dyn[];
    int* s_sub = s_dyn;           // [8][E]: per-warp counts, then per-warp bases
    int* s_ids = s_dyn + 8 * E;   // [8][32 k]: each warp's slot experts
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    ptx::griddep_launch_dependents();
    const int nb = (T + kCountTokens - 1) / kCountTokens;
    if (static_cast<int>(blockIdx.x) >= nb) {
        const int t = (static_cast<int>(blockIdx.x) - nb) * kRouteWarps + warp;
        if (t < T) {
            GateLogit gl;
            gl.load(t, H, hidden, w_g, lane, 0);
            const float z = gl.finish(t, H, hidden, w_g, lane);
            if (lane == 0) gate_logit[t] = z;
        }
        return;
    }
    for (int i = tid; i < 8 * E; i += 256) s_sub[i] = 0;
    __syncthreads();
    ptx::griddep_wait();
    const long t0 = static_cast<long>(blockIdx.x) * kCountTokens + warp * 32;
    const long t1 = min(static_cast<long>(T), t0 + 32);
    const long wa0 = t0 * k, wa1 = t1 > t0 ? t1 * k : wa0;
    const int n = static_cast<int>(wa1 - wa0);  // <= 32 k
    int* ids = s_ids + warp * 32 * k;
    // The warp's slot experts are read once (all loads in flight together)
    // and both passes below work from shared memory.
#pragma unroll 8
    for (int i = lane; i < n; i += 32) ids[i] = topk_ids[wa0 + i];
    __syncwarp();
    int* running = s_sub + warp * E;
    for (int i = lane; i < n; i += 32) atomicAdd(&running[ids[i]], 1);
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
    ordered_scatter(ids, wa0, wa1, running, perm, inv, lane);
}

__global__ void __launch_bounds__(256)
combine_kernel(int T, int H, int k, const float* __restrict__ y, const float* __restrict__ y_shared,
               const float* __restrict__ topk_w, const int* __restrict__ inv,
               __nv_bfloat16* __restrict__ out) {
    const int t = blockIdx.x;
    const int h = (blockIdx.y * 256 + threadIdx.x) * 4;
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
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
    const float4 s = __ldcs(reinterpret_cast<const float4*>(y_shared + static_cast<size_t>(t) * H + h));
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

// The same combine over y stored as y16 codes (2H-byte rows, then one
// exponent byte per 32 values of each row in the exponent plane). A thread
// owns 16 consecutive outputs (combine16_y16): per row it reads 32
// contiguous bytes of codes (a warp: 1 KB) and the exponent byte of their
// block. CTAs of 256 threads cover 256 / (H/16) whole tokens (two at H =
// 2048), or with H/16 > 256 one token's outputs over gridDim.y CTAs.
__global__ void __launch_bounds__(256)
combine_y16_kernel(int T, int H, int k, const uint8_t* __restrict__ y,
                   const float* __restrict__ topk_w, const int* __restrict__ inv,
                   __nv_bfloat16* __restrict__ out) {
    const int per = min(H / 16, 256);  // threads per token and CTA (H is a multiple of 64)
    const int tpc = 256 / per;         // tokens per CTA
    const int t = blockIdx.x * tpc + static_cast<int>(threadIdx.x) / per;
    const int h = (blockIdx.y * 256 + static_cast<int>(threadIdx.x) % per) * 16;
    if (t >= T || static_cast<int>(threadIdx.x) >= tpc * per || h >= H) return;
    combine16_y16(t, h, T, H, k, y, topk_w, inv, out);
}

// fp32 values through the y16 format (the down GEMMs' encoder, the combine's
// decoder): warp w takes blocks w, w + warps, ... of 32 values, lane i value
// i; the block's exponent byte comes from a warp-wide maximum, as in the
// weights-on-M down epilogue.
__global__ void __launch_bounds__(256)
y16_roundtrip_kernel(long n, const float* __restrict__ in, float* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const long warps = static_cast<long>(gridDim.x) * 8;
    for (long blk = static_cast<long>(blockIdx.x) * 8 + (threadIdx.x >> 5); blk * 32 < n; blk += warps) {
        const uint32_t x = __float_as_uint(in[blk * 32 + lane]);
        const uint32_t b = y16_block_exp(__reduce_max_sync(0xFFFFFFFFu, x & 0x7FFFFFFFu));
        out[blk * 32 + lane] = y16_decode(y16_encode(x, b), b);
    }
}

// ---------------------------------------------------- expert parallelism
// Rows of the (token, slot) pairs in expert-sorted order: rows[p] =
// hidden[perm[p] / k]. The rows bound for one rank's block of experts are
// then one contiguous range (the send buffer of the dispatch exchange).
__global__ void __launch_bounds__(256)
gather_rows_kernel(int H, int k, const int* __restrict__ perm,
                   const __nv_bfloat16* __restrict__ hidden, __nv_bfloat16* __restrict__ rows) {
    const int p = blockIdx.x;
    const int c = blockIdx.y * 256 + threadIdx.x;  // 16-byte chunk of the row
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    if (c >= H / 8) return;
    const int t = perm[p] / k;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(hidden + static_cast<size_t>(t) * H) + c);
    reinterpret_cast<uint4*>(rows + static_cast<size_t>(p) * H)[c] = v;
}

// Row tiles of the rows one rank received in the dispatch exchange: G source
// segments in source order, each holding its rows sorted by local expert, with
// recv_counts[s * E_loc + e] rows of expert e from source s. Thread i owns
// segment i (i = s * E_loc + e); the segments' rows and tiles are exclusive
// scans in that order. Tiles are {local expert, first row in the segment,
// rows, first row in the received buffer}. If the counts are negative or do
// not add up to R, no routed tile is written and the status word records
// ERR_EP_COUNTS (the shared expert's tiles still run).
__global__ void __launch_bounds__(kEpTileThreads)
ep_tiles_kernel(int G, int E_loc, int R, const int* __restrict__ recv_counts, int bn_gu,
                int bn_dn, int4* __restrict__ rt_gu, int4* __restrict__ rt_dn,
                int* __restrict__ meta) {
    constexpr int NW = kEpTileThreads / 32;
    __shared__ int s_warp[NW];
    __shared__ int s_off[kMaxExperts + 1];
    __shared__ int s_tstart[kMaxExperts + 1];
    __shared__ int s_bad;
    const int tid = threadIdx.x;
    const int nseg = G * E_loc;  // <= kMaxExperts
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    if (tid == 0) s_bad = 0;
    __syncthreads();
    const int c = tid < nseg ? recv_counts[tid] : 0;
    if (c < 0) atomicOr(&s_bad, 1);
    int total;
    const int off = block_excl_scan<NW>(c < 0 ? 0 : c, s_warp, &total);
    if (tid < nseg) s_off[tid] = off;
    if (tid == 0) s_off[nseg] = total;
    __syncthreads();
    const bool bad = s_bad != 0 || total != R;
    if (bad) {
        if (tid == 0) {
            meta[META_RT_GU] = 0;
            meta[META_RT_DN] = 0;
            atomicOr(reinterpret_cast<unsigned*>(meta + META_ERR), ERR_EP_COUNTS);
        }
        return;
    }
    for (int g = 0; g < 2; ++g) {
        const int bn = g == 0 ? bn_gu : bn_dn;
        int tot_tiles;
        const int pos = block_excl_scan<NW>((c + bn - 1) / bn, s_warp, &tot_tiles);
        if (tid < nseg) s_tstart[tid] = pos;
        if (tid == 0) s_tstart[nseg] = tot_tiles;
        __syncthreads();
        int4* rt = g == 0 ? rt_gu : rt_dn;
        for (int i = tid; i < tot_tiles; i += kEpTileThreads) {
            int lo = 0, hi = nseg - 1;  // the largest segment with s_tstart <= i
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_tstart[mid] <= i) lo = mid;
                else hi = mid - 1;
            }
            const int m0 = (i - s_tstart[lo]) * bn;
            const int n = s_off[lo + 1] - s_off[lo];
            rt[i] = make_int4(lo % E_loc, m0, min(bn, n - m0), s_off[lo] + m0);
        }
        if (tid == 0) meta[g == 0 ? META_RT_GU : META_RT_DN] = tot_tiles;
        __syncthreads();
    }
}

}  // namespace

bool route_small_fits(int T, int E, int k) {
    return static_cast<long>(T) * k <= kSmallSlots && E <= 1024;
}

namespace {
int experts_per_lane(int E) {
    int epl = 1;
    while (32 * epl < E) epl *= 2;
    return epl;  // 1 .. 32 for E <= 1024
}
}  // namespace

#define MOE_EPL_DISPATCH(EPLV, CALL) \
    switch (EPLV) {                  \
        case 1: CALL(1);             \
        case 2: CALL(2);             \
        case 4: CALL(4);             \
        case 8: CALL(8);             \
        case 16: CALL(16);           \
        default: CALL(32);           \
    }

cudaError_t launch_route_permute(int T, int H, int E, int k, int score_fn, int bn_gu, int bn_dn,
                                 const LogitSrc& logits, bool pdl, const __nv_bfloat16* hidden,
                                 const __nv_bfloat16* w_g, int* topk_ids, float* topk_w,
                                 float* gate_logit, int* counts, int* offsets, int* perm,
                                 int* inv, int4* rt_gu, int4* rt_dn, int* meta, int* ids_out,
                                 float* w_out, int* counts_out, cudaStream_t st) {
    const int blocks = T;  // one token per CTA
    const size_t smem = (static_cast<size_t>(T) * k + static_cast<size_t>(kRouteWarps) * E) *
                        sizeof(int);
#define MOE_LAUNCH_RP(N)                                                                        \
    return launch_kernel(route_permute_kernel<N>, dim3(blocks), dim3(kRouteWarps * 32), smem,  \
                         st, pdl, T, H, E, k, score_fn, bn_gu, bn_dn, logits, hidden, w_g,      \
                         topk_ids, topk_w, gate_logit, counts, offsets, perm, inv, rt_gu, rt_dn, \
                         meta, ids_out, w_out, counts_out)
    MOE_EPL_DISPATCH(experts_per_lane(E), MOE_LAUNCH_RP)
#undef MOE_LAUNCH_RP
}

cudaError_t launch_route_count(int T, int E, int k, int score_fn, int bn_gu, int bn_dn,
                               const LogitSrc& logits, bool pdl, int* topk_ids, float* topk_w,
                               int* blockhist, int* counts, int* offsets, int4* rt_gu, int4* rt_dn,
                               int* meta, int* ids_out, float* w_out, int* counts_out,
                               cudaStream_t st) {
    const int blocks = (T + kRouteWarps - 1) / kRouteWarps;
#define MOE_LAUNCH_RC(N)                                                                        \
    return launch_kernel(route_count_kernel<N>, dim3(blocks), dim3(kRouteWarps * 32), 0, st,  \
                         pdl, T, E, k, score_fn, bn_gu, bn_dn, logits, topk_ids, topk_w,         \
                         blockhist, counts, offsets, rt_gu, rt_dn, meta, ids_out, w_out,         \
                         counts_out)
    MOE_EPL_DISPATCH(experts_per_lane(E), MOE_LAUNCH_RC)
#undef MOE_LAUNCH_RC
}

cudaError_t launch_scatter(int T, int H, int E, int k, const int* topk_ids, const int* blockhist,
                           const int* offsets, int* perm, int* inv, const __nv_bfloat16* hidden,
                           const __nv_bfloat16* w_g, float* gate_logit, cudaStream_t st) {
    const int blocks =
        (T + kCountTokens - 1) / kCountTokens + (T + kRouteWarps - 1) / kRouteWarps;
    const size_t smem = (8 * static_cast<size_t>(E) + 8 * 32 * static_cast<size_t>(k)) * sizeof(int);
    if (smem > 48 * 1024) {  // E = 1024 with k = 32 needs 64 KB
        const cudaError_t e = cudaFuncSetAttribute(
            scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(scatter_kernel, dim3(blocks), dim3(256), smem, st, true, T, H, E, k,
                         topk_ids, blockhist, offsets, perm, inv, hidden, w_g, gate_logit);
}

cudaError_t launch_combine(int T, int H, int k, const float* y, bool y16, const float* topk_w,
                           const int* inv, __nv_bfloat16* out, cudaStream_t st) {
    if (y16) {
        // An ordinary launch, after the down GEMM has finished: as a programmatic
        // dependent its CTAs would sit resident beside the down GEMM's CTAs for
        // all of that kernel, and the step measured 1-3 % slower (prefill, skewed,
        // wide) than with this launch.
        const int per = H / 16 < 256 ? H / 16 : 256, tpc = 256 / per;
        dim3 grid((T + tpc - 1) / tpc, (H / 16 + 255) / 256);
        return launch_kernel(combine_y16_kernel, grid, dim3(256), 0, st, false, T, H, k,
                             reinterpret_cast<const uint8_t*>(y), topk_w, inv, out);
    }
    dim3 grid(T, (H / 4 + 255) / 256);
    return launch_kernel(combine_kernel, grid, dim3(256), 0, st, true, T, H, k, y,
                         y + static_cast<size_t>(T) * k * H, topk_w, inv, out);
}

cudaError_t launch_y16_roundtrip(long n, const float* in, float* out, cudaStream_t st) {
    const long blocks = (n / 32 + 7) / 8;
    y16_roundtrip_kernel<<<static_cast<unsigned>(blocks < 1184 ? blocks : 1184), 256, 0, st>>>(n, in, out);
    return cudaGetLastError();
}

cudaError_t launch_combine_split(int T, int H, int k, const float* y_routed, const float* y_shared,
                                 const float* topk_w, const int* inv, __nv_bfloat16* out,
                                 cudaStream_t st) {
    dim3 grid(T, (H / 4 + 255) / 256);
    return launch_kernel(combine_kernel, grid, dim3(256), 0, st, true, T, H, k, y_routed, y_shared,
                         topk_w, inv, out);
}

cudaError_t launch_gather_rows(int P, int H, int k, const int* perm,
                               const __nv_bfloat16* hidden, __nv_bfloat16* rows, cudaStream_t st) {
    if (P == 0) return cudaSuccess;
    dim3 grid(P, (H / 8 + 255) / 256);
    return launch_kernel(gather_rows_kernel, grid, dim3(256), 0, st, true, H, k, perm, hidden,
                         rows);
}

cudaError_t launch_ep_tiles(int G, int E_loc, int R, const int* recv_counts, int bn_gu,
                            int bn_dn, int4* rt_gu, int4* rt_dn, int* meta, cudaStream_t st) {
    return launch_kernel(ep_tiles_kernel, dim3(1), dim3(kEpTileThreads), 0, st, true, G, E_loc, R,
                         recv_counts, bn_gu, bn_dn, rt_gu, rt_dn, meta);
}

}  // namespace moe
