// Routing device code shared by the routing kernels (moe_route.cu) and the
// whole-layer fused launch (moe_fused.cu): the per-token score, top-k and
// renormalisation, the gate logit, and the small-batch permute.
//
//   routing     per token: score, top-k (ties to the lower expert index),
//               renormalisation, and the shared-expert gate logit x . w_g.
//               Router in fp32, softmax or sigmoid score, normalised top-k
//               affinities: "Add Qwen3.5-35B-A3B (support vision and text
//               input)", Model Information and Additional Information.
//   permute     per-expert counts, exclusive offsets, the stable expert-sorted
//               order of (token, slot) pairs (tokens ascending within an
//               expert), its inverse, and the row-tile lists of both grouped
//               GEMMs. Each row tile is {expert, first row, rows, first
//               sorted position}.
#pragma once

#include "moe_internal.cuh"
#include "ptx.cuh"

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

// Logit value of a key (inverse of rank_key on canonical values).
__device__ __forceinline__ float key_value(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
}

// One 64-bit code per (logit, expert): larger code ranks first; for equal
// logits the lower expert index has the larger code. Codes are distinct and
// nonzero for e < 2^32 - 1.
__device__ __forceinline__ uint64_t rank_code(float v, int e) {
    return (static_cast<uint64_t>(rank_key(v)) << 32) |
           static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(e));
}

// Routing of one token by one warp; lane i holds the logits of experts i,
// i+32, ... (EPL of them, E <= 32*EPL). Each round takes the warp-wide best of
// the lanes' current bests; only the lane that supplied it looks for its next
// best. Lane j < k returns the j-th selected expert and its renormalised weight.
template <int EPL>
__device__ __forceinline__ void route_token(const float (&v)[EPL], int E, int k, int score_fn,
                                            int lane, int& my_e, float& my_w) {
    uint64_t c[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        c[i] = e < E ? rank_code(v[i], e) : 0ull;
    }
    uint64_t lane_best = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) lane_best = c[i] > lane_best ? c[i] : lane_best;
    uint64_t mine = 0;
    for (int j = 0; j < k; ++j) {
        // Warp-wide maximum of the 64-bit codes: the largest logit key first;
        // when one lane holds it (the usual case) its code is the maximum,
        // otherwise the largest inverted index among the tied lanes decides.
        const uint32_t key = static_cast<uint32_t>(lane_best >> 32);
        const uint32_t khi = __reduce_max_sync(0xFFFFFFFFu, key);
        const unsigned tied = __ballot_sync(0xFFFFFFFFu, key == khi);
        uint32_t klo;
        if ((tied & (tied - 1u)) == 0u)
            klo = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(lane_best), __ffs(tied) - 1);
        else
            klo = __reduce_max_sync(0xFFFFFFFFu,
                                    key == khi ? static_cast<uint32_t>(lane_best) : 0u);
        const uint64_t best = (static_cast<uint64_t>(khi) << 32) | klo;
        if (lane == j) mine = best;
        if (lane_best == best) {
            uint64_t nb = 0;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (c[i] < best && c[i] > nb) nb = c[i];
            lane_best = nb;
        }
    }
    my_e = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(mine));
    const float my_v = key_value(static_cast<uint32_t>(mine >> 32));
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
    my_w = s / sum;
}

// Shared-expert gate logit z_t = x_t . w_g, fp32 accumulation, by one warp.
// The row is read in batches of kGateBatch 16-byte chunks per lane: load()
// issues the first batch early (its latency overlaps the top-k selection) and
// finish() consumes it and any further batches. Lane i accumulates chunks
// i, i+32, ... in order, then the warp sums the lanes.
constexpr int kGateBatch = 4;

struct GateLogit {
    uint4 x[kGateBatch], g[kGateBatch];

    __device__ __forceinline__ void load(int t, int H, const __nv_bfloat16* __restrict__ hidden,
                                         const __nv_bfloat16* __restrict__ w_g, int lane, int c0) {
        const uint4* xr = reinterpret_cast<const uint4*>(hidden + static_cast<size_t>(t) * H);
        const uint4* gr = reinterpret_cast<const uint4*>(w_g);
        const int nch = H / 8;
#pragma unroll
        for (int i = 0; i < kGateBatch; ++i) {
            const int c = c0 + lane + 32 * i;
            if (c < nch) {
                x[i] = __ldcs(xr + c);
                g[i] = __ldg(gr + c);
            } else {
                x[i] = make_uint4(0u, 0u, 0u, 0u);
                g[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }

    __device__ __forceinline__ float dot(float acc) const {
#pragma unroll
        for (int i = 0; i < kGateBatch; ++i) {
            const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&x[i]);
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&g[i]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 fa = __bfloat1622float2(a2[q]);
                const float2 fb = __bfloat1622float2(b2[q]);
                acc = fmaf(fa.x, fb.x, acc);
                acc = fmaf(fa.y, fb.y, acc);
            }
        }
        return acc;
    }

    // Chunks past the row end were loaded as zeros and add exact zeros.
    __device__ __forceinline__ float finish(int t, int H, const __nv_bfloat16* __restrict__ hidden,
                                            const __nv_bfloat16* __restrict__ w_g, int lane) {
        float acc = dot(0.f);
        for (int c0 = 32 * kGateBatch; c0 < H / 8; c0 += 32 * kGateBatch) {
            load(t, H, hidden, w_g, lane, c0);
            acc = dot(acc);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
        return acc;
    }
};

// Exclusive scan of one int per thread over a block of NW warps; *total gets
// the block sum. Contains __syncthreads: every thread must call it.
template <int NW>
__device__ int block_excl_scan(int v, int* s_warp, int* total) {
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
    for (int w = 0; w < NW; ++w) {
        const int x = s_warp[w];
        if (w < warp) base += x;
        tot += x;
    }
    *total = tot;
    return base + incl - v;
}

// The same scan among the first NW warps of the CTA only, synchronised with
// named barrier 1 (the other warps of the CTA may be elsewhere).
template <int NW>
__device__ int bar_excl_scan(int v, int* s_warp, int* total) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    ptx::named_bar_sync(1, NW * 32);
    if (lane == 31) s_warp[warp] = incl;
    ptx::named_bar_sync(1, NW * 32);
    int base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const int x = s_warp[w];
        if (w < warp) base += x;
        tot += x;
    }
    *total = tot;
    return base + incl - v;
}

// Row tiles of one expert: {expert, first row, rows, first sorted position}.
__device__ __forceinline__ void write_row_tiles(int4* rt, int pos, int e, int n_e, int off_e,
                                                int bn) {
    for (int m0 = 0; m0 < n_e; m0 += bn)
        rt[pos++] = make_int4(e, m0, min(bn, n_e - m0), off_e + m0);
}

// Ordered (stable) scatter of the slots [a0, a1) by one warp; the expert of
// slot a is ids[a - a0] and `running[e]` is the next free sorted position of
// expert e. Equal experts inside a 32-slot chunk are ranked by lane, so slot
// order (token order) is kept.
__device__ __forceinline__ void ordered_scatter(const int* ids, long a0, long a1, int* running,
                                                int* __restrict__ perm, int* __restrict__ inv,
                                                int lane) {
    for (long base = a0; base < a1; base += 32) {
        const long a = base + lane;
        const int e = a < a1 ? ids[a - a0] : -1;
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

// Routing of one token per warp; writes ids, weights and (with GATE) the gate
// logit. Lane j < k returns the token's j-th selected expert.
template <int EPL, bool GATE = true>
__device__ __forceinline__ int route_and_store(int t, int H, int E, int k, int score_fn,
                                                const LogitSrc& logits,
                                                const __nv_bfloat16* __restrict__ hidden,
                                                const __nv_bfloat16* __restrict__ w_g,
                                                int* __restrict__ topk_ids,
                                                float* __restrict__ topk_w,
                                                float* __restrict__ gate_logit,
                                                int* __restrict__ ids_out,
                                                float* __restrict__ w_out, int lane) {
    // All loads are issued first: the hidden row's latency overlaps the top-k.
    const float* lg = logits.p + static_cast<size_t>(t) * E;
    float v[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? __ldcs(lg + e) : 0.f;
    }
    if (logits.parts > 1) {  // split-K partial sums of the router GEMM, added in order
        for (int s = 1; s < logits.parts; ++s) {
            const float* ls = lg + static_cast<size_t>(s) * logits.part_stride;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = lane + 32 * i;
                if (e < E) v[i] += __ldcs(ls + e);
            }
        }
    }
    if (logits.out) {
        float* lo = logits.out + static_cast<size_t>(t) * E;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) lo[e] = v[i];
        }
    }
    GateLogit gl;
    if (GATE) gl.load(t, H, hidden, w_g, lane, 0);
    int my_e;
    float my_w;
    route_token<EPL>(v, E, k, score_fn, lane, my_e, my_w);
    if (GATE) {
        const float z = gl.finish(t, H, hidden, w_g, lane);
        if (lane == 0) gate_logit[t] = z;
    }
    if (lane < k) {
        const size_t o = static_cast<size_t>(t) * k + lane;
        topk_ids[o] = my_e;
        topk_w[o] = my_w;
        if (ids_out) ids_out[o] = my_e;
        if (w_out) w_out[o] = my_w;
    }
    return my_e;
}

// ------------------------------------------------------------ small batches
// Threads of the small-batch routing: the CTA's first kRouteWarps warps (the
// whole CTA of the routing kernel; part of the whole-layer launch's CTA).
constexpr int kSmallThreads = kRouteWarps * 32;

// Routing of token t by the first kSmallThreads threads of the CTA: warp 0
// selects the experts and writes ids and weights; the eight warps share the
// gate logit z_t = x_t . w_g. Thread i takes the 16-byte chunks i, i + 256,
// ... of the row, loaded before warp 0's top-k so that their latency overlaps
// it; the threads' sums are added per warp, then in warp order. Synchronises
// those threads (named barrier 1) and leaves s_gate free for the next token.
template <int EPL>
__device__ __forceinline__ void route_token_cta(int t, int H, int E, int k, int score_fn,
                                                const LogitSrc& logits,
                                                const __nv_bfloat16* __restrict__ hidden,
                                                const __nv_bfloat16* __restrict__ w_g,
                                                int* __restrict__ topk_ids,
                                                float* __restrict__ topk_w,
                                                float* __restrict__ gate_logit,
                                                int* __restrict__ ids_out,
                                                float* __restrict__ w_out, float* s_gate) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint4* xr = reinterpret_cast<const uint4*>(hidden + static_cast<size_t>(t) * H);
    const uint4* gr = reinterpret_cast<const uint4*>(w_g);
    const int nch = H / 8;
    uint4 xa[kGateBatch], ga[kGateBatch];
    auto load = [&](int c0) {
#pragma unroll
        for (int i = 0; i < kGateBatch; ++i) {
            const int c = c0 + tid + kSmallThreads * i;
            xa[i] = c < nch ? __ldcs(xr + c) : make_uint4(0u, 0u, 0u, 0u);
            ga[i] = c < nch ? __ldg(gr + c) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    load(0);
    if (warp == 0)
        route_and_store<EPL, false>(t, H, E, k, score_fn, logits, hidden, w_g, topk_ids, topk_w,
                                    gate_logit, ids_out, w_out, lane);
    float acc = 0.f;
    for (int c0 = 0; c0 < nch; c0 += kSmallThreads * kGateBatch) {
        if (c0 > 0) load(c0);
#pragma unroll
        for (int i = 0; i < kGateBatch; ++i) {
            const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&xa[i]);
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&ga[i]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 fa = __bfloat1622float2(a2[q]);
                const float2 fb = __bfloat1622float2(b2[q]);
                acc = fmaf(fa.x, fb.x, acc);
                acc = fmaf(fa.y, fb.y, acc);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) s_gate[warp] = acc;
    ptx::named_bar_sync(1, kSmallThreads);
    if (tid == 0) {
        float z = 0.f;
#pragma unroll
        for (int w = 0; w < kRouteWarps; ++w) z += s_gate[w];
        gate_logit[t] = z;
    }
    ptx::named_bar_sync(1, kSmallThreads);
}

// The complete permute of T*k <= kSmallSlots slots by the first kSmallThreads
// threads of one CTA, once every token is routed (topk_ids written and
// visible): counts, offsets, both GEMMs' row tiles and their tile counts in
// meta, the stable sorted order perm and its inverse inv. Warp w owns the
// contiguous slot range [a0_w, a1_w). s_scr holds T*k + kRouteWarps*E ints,
// s_warp kRouteWarps ints.
__device__ __forceinline__ void permute_small(int T, int E, int k, int bn_gu, int bn_dn,
                                              const int* __restrict__ topk_ids,
                                              int* __restrict__ counts, int* __restrict__ offsets,
                                              int* __restrict__ perm, int* __restrict__ inv,
                                              int4* __restrict__ rt_gu, int4* __restrict__ rt_dn,
                                              int* __restrict__ meta,
                                              int* __restrict__ counts_out, int* s_scr,
                                              int* s_warp) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tk = T * k;
    int* s_ids = s_scr;              // [T*k]
    int* s_sub = s_scr + tk;         // [kRouteWarps][E]: per-warp counts, then bases
    for (int a = tid; a < tk; a += kSmallThreads) s_ids[a] = __ldcg(&topk_ids[a]);
    for (int i = tid; i < kRouteWarps * E; i += kSmallThreads) s_sub[i] = 0;
    ptx::named_bar_sync(1, kSmallThreads);
    const int chunk = (tk + kRouteWarps - 1) / kRouteWarps;
    const int a0 = min(tk, warp * chunk), a1 = min(tk, a0 + chunk);
    for (int a = a0 + lane; a < a1; a += 32) atomicAdd(&s_sub[warp * E + s_ids[a]], 1);
    ptx::named_bar_sync(1, kSmallThreads);
    // Thread tid owns experts [tid*ept, tid*ept + ept): totals, then a scan.
    const int ept = (E + kSmallThreads - 1) / kSmallThreads;  // <= 4
    int local[4] = {0, 0, 0, 0};
    int mine = 0;
    for (int r = 0; r < ept; ++r) {
        const int e = tid * ept + r;
        if (e >= E) break;
        int c = 0;
        for (int w = 0; w < kRouteWarps; ++w) c += s_sub[w * E + e];
        local[r] = c;
        mine += c;
    }
    int total;
    const int first_off = bar_excl_scan<kRouteWarps>(mine, s_warp, &total);
    int run = first_off;
    for (int r = 0; r < ept; ++r) {
        const int e = tid * ept + r;
        if (e >= E) break;
        counts[e] = local[r];
        offsets[e] = run;
        if (counts_out) counts_out[e] = local[r];
        int b = run;  // per-warp bases inside expert e, in warp (= slot) order
        for (int w = 0; w < kRouteWarps; ++w) {
            const int v = s_sub[w * E + e];
            s_sub[w * E + e] = b;
            b += v;
        }
        run += local[r];
    }
    if (tid == 0) offsets[E] = total;
    for (int g = 0; g < 2; ++g) {
        const int bn = g == 0 ? bn_gu : bn_dn;
        int nt = 0;
        for (int r = 0; r < ept; ++r) nt += (local[r] + bn - 1) / bn;
        int tot_tiles;
        int pos = bar_excl_scan<kRouteWarps>(nt, s_warp, &tot_tiles);
        int off = first_off;
        for (int r = 0; r < ept; ++r) {
            const int e = tid * ept + r;
            if (e >= E) break;
            write_row_tiles(g == 0 ? rt_gu : rt_dn, pos, e, local[r], off, bn);
            pos += (local[r] + bn - 1) / bn;
            off += local[r];
        }
        if (tid == 0) meta[g == 0 ? META_RT_GU : META_RT_DN] = tot_tiles;
    }
    ptx::named_bar_sync(1, kSmallThreads);
    ordered_scatter(s_ids + a0, a0, a1, s_sub + warp * E, perm, inv, lane);
}

// 16 consecutive values of one y16 row (codes at `codes`, their block's
// exponent byte at `exps`).
__device__ __forceinline__ void y16_row16(const uint8_t* __restrict__ codes,
                                          const uint8_t* __restrict__ exps, float (&f)[16]) {
    const uint4* c = reinterpret_cast<const uint4*>(codes);
    const uint4 c0 = __ldcs(c), c1 = __ldcs(c + 1);
    const uint32_t b = __ldcs(exps);
    const uint32_t wv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f[2 * i] = y16_decode(wv[i] & 0xFFFFu, b);
        f[2 * i + 1] = y16_decode(wv[i] >> 16, b);
    }
}

// out[t, h .. h+15] = bf16(sum_j w_tj y[inv(t,j)] + y[T k + t]) over y16
// rows (T k routed rows in sorted order, then T gated shared rows; codes
// from y, then the exponent plane), summed in fp32 in slot order with one
// rounding. h is a multiple of 16 below H (a multiple of 64).
__device__ __forceinline__ void combine16_y16(int t, int h, int T, int H, int k,
                                              const uint8_t* __restrict__ y,
                                              const float* __restrict__ topk_w,
                                              const int* __restrict__ inv,
                                              __nv_bfloat16* __restrict__ out) {
    const size_t rows = static_cast<size_t>(T) * k + T;
    const size_t row_bytes = 2 * static_cast<size_t>(H);
    const uint8_t* codes = y + 2 * static_cast<size_t>(h);
    const uint8_t* exps = y + rows * row_bytes + h / kY16Block;
    const size_t es = static_cast<size_t>(y16_exp_stride(H));
    const size_t tk = static_cast<size_t>(t) * k;
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll 4
    for (int j = 0; j < k; ++j) {
        const float w = topk_w[tk + j];
        const size_t p = static_cast<size_t>(inv[tk + j]);
        float f[16];
        y16_row16(codes + p * row_bytes, exps + p * es, f);
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = fmaf(w, f[i], acc[i]);
    }
    {
        const size_t p = static_cast<size_t>(T) * k + t;
        float f[16];
        y16_row16(codes + p * row_bytes, exps + p * es, f);
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] += f[i];
    }
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        o[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H + h);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// out_t = bf16(sum_j w_tj y[inv(t,j)] + y_shared[t]) for one token, summed in
// fp32 in slot order; thread i of nthreads takes 4 columns at a time from 4i.
// The arithmetic is the combine kernel's (fp32 y).
__device__ __forceinline__ void combine_token(int t, int H, int k, const float* __restrict__ y,
                                              const float* __restrict__ y_shared,
                                              const float* __restrict__ topk_w,
                                              const int* __restrict__ inv,
                                              __nv_bfloat16* __restrict__ out, int tid,
                                              int nthreads) {
    const size_t tk = static_cast<size_t>(t) * k;
    for (int h = tid * 4; h < H; h += nthreads * 4) {
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
}

}  // namespace
}  // namespace moe
