// Router logits on the FFN side: logits[t][e] = sum_h x[t][h] W_router[e][h],
// with W_router [E, H] bf16 and fp32 accumulation (the router runs in fp32:
// "Add Qwen3.5-35B-A3B (support vision and text input)", Additional
// Information; products of bf16 values are exact in fp32).
//
// A split-K tcgen05 GEMM: CTA (m, n, s) computes the 128 experts m*128.. of
// the BN tokens n*BN.. over the s-th of S ranges of 64-value K steps, D[128,
// BN] = W_router_tile X_tile^T in TMEM, and writes that partial sum to
// partial[s]; the routing kernels, launched as its programmatic dependents,
// add the S partials of every logit in the fixed order s = 0..S-1 as they
// load them (no atomics: the logits, and so the routing, are the same on
// every run). S is chosen so that a decode-sized batch (a few output tiles)
// still spreads over tens of SMs.
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 TMEM owner and MMA
// issuer, warps 2-5 epilogue (warp w drains TMEM lane quadrant w % 4: 32
// experts, one per lane, so a warp's stores of one token are 128 contiguous
// bytes). Waits are bounded as in the expert GEMMs.
#include "gemm_common.cuh"

namespace moe {
namespace {

constexpr int kRouterThreads = 192;
constexpr int kRouterStages = 4;

template <int BN>
struct RouterCfg {
    static constexpr int A_BYTES = kGemmBM * kGemmBK * 2;  // 16 KB of W_router rows
    static constexpr int B_BYTES = BN * kGemmBK * 2;       // token rows
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int CTL_OFF = kRouterStages * STAGE_BYTES;
    static constexpr int SMEM = 1024 + CTL_OFF + 1024;
    static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;
    static_assert(SMEM <= kSmemLimit, "shared memory budget");
    static_assert(BN % 16 == 0 && BN <= 256 && (BN & (BN - 1)) == 0, "MMA N, TMEM allocation");
};

struct RouterCtl {
    uint64_t full[kRouterStages];
    uint64_t empty[kRouterStages];
    uint64_t done;  // accumulator complete (and the abort-path drain)
    uint32_t tmem_base;
    int abort;
};

template <int BN>
__global__ void __launch_bounds__(kRouterThreads, 1)
router_gemm_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                   int T, int H, int E, int S, float* __restrict__ out, unsigned* err) {
    using C = RouterCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    RouterCtl* ctl = reinterpret_cast<RouterCtl*>(smem + C::CTL_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ptx::griddep_launch_dependents();  // the routing CTAs may start their set-up
    const int m0 = blockIdx.x * kGemmBM, n0 = blockIdx.y * BN, split = blockIdx.z;
    const int ksteps = H / kGemmBK;
    const int k_begin = static_cast<int>(static_cast<long long>(ksteps) * split / S);
    const int k_end = static_cast<int>(static_cast<long long>(ksteps) * (split + 1) / S);
    volatile int* abort_flag = &ctl->abort;
    const unsigned code = ERR_ROUTER_TIMEOUT;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRouterStages; ++s) {
            ptx::mbar_init(bar_addr(&ctl->full[s]), 1);
            ptx::mbar_init(bar_addr(&ctl->empty[s]), 1);
        }
        ptx::mbar_init(bar_addr(&ctl->done), 1);
        ctl->abort = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&map_w);
        ptx::prefetch_tmap(&map_x);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&ctl->tmem_base), C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;

    if (warp == 0) {
        if (lane == 0) {  // ---------------------------------- TMA producer
            const uint64_t pol = ptx::policy_evict_last();  // W_router is re-read by every token tile
            int s = 0;
            uint32_t ph = 0, armed = 0, parity_bits = 0;
            bool ok = true;
            for (int ks = k_begin; ks < k_end; ++ks) {
                if (!wait_bar(bar_addr(&ctl->empty[s]), ph ^ 1u, abort_flag, err, code)) {
                    ok = false;
                    break;
                }
                const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
                const uint32_t fb = bar_addr(&ctl->full[s]);
                ptx::mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
                ptx::tma_load_2d(sa, &map_w, fb, ks * kGemmBK, m0, pol);
                ptx::tma_load_2d(sa + C::A_BYTES, &map_x, fb, ks * kGemmBK, n0, pol);
                armed |= 1u << s;
                parity_bits = (parity_bits & ~(1u << s)) | (ph << s);
                if (++s == kRouterStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok)  // no copy may still be in flight when the CTA exits
                for (int i = 0; i < kRouterStages; ++i)
                    if (armed & (1u << i)) wait_bounded(bar_addr(&ctl->full[i]), (parity_bits >> i) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------------------------- MMA issuer
            const uint32_t idesc = ptx::idesc_bf16_f32(kGemmBM, BN);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int ks = k_begin; ks < k_end; ++ks) {
                if (!wait_bar(bar_addr(&ctl->full[s]), ph, abort_flag, err, code)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
                const uint64_t da = ptx::smem_desc_sw128(sa);
                const uint64_t db = ptx::smem_desc_sw128(sa + C::A_BYTES);
#pragma unroll
                for (int kk = 0; kk < kGemmBK / 16; ++kk)
                    ptx::mma_bf16_ss(tmem_base, da + 2 * kk, db + 2 * kk, idesc,
                                     (ks > k_begin || kk > 0) ? 1u : 0u);
                ptx::mma_commit(bar_addr(&ctl->empty[s]));
                if (++s == kRouterStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // Signals the epilogue; on the abort path the epilogue's wait sees the
            // abort flag instead, and this commit still drains the issued MMAs.
            ptx::mma_commit(bar_addr(&ctl->done));
            if (!ok) wait_bounded(bar_addr(&ctl->done), 0);
        }
    } else {  // ------------------------------------------- epilogue (warps 2-5)
        const int q = warp & 3;
        const int e = m0 + q * 32 + lane;
        if (wait_bar(bar_addr(&ctl->done), 0, abort_flag, err, code)) {
            ptx::tc_fence_after();
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            float* dst = out + static_cast<size_t>(split) * T * E;
            for (int c0 = 0; c0 < BN; c0 += 16) {
                if (n0 + c0 >= T) break;
                uint32_t v[16];
                ptx::tmem_ld_32x32b_x16(tb + c0, v);
                ptx::tmem_ld_wait();
                if (e < E) {  // every K range has at least one step, so D is written
#pragma unroll
                    for (int n = 0; n < 16; ++n) {
                        const int t = n0 + c0 + n;
                        if (t < T) dst[static_cast<size_t>(t) * E + e] = __uint_as_float(v[n]);
                    }
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int BN>
cudaError_t launch_router_bn(const CUtensorMap& map_w, const CUtensorMap& map_x, int T, int H,
                             int E, int S, float* out, unsigned* err, cudaStream_t st) {
    using C = RouterCfg<BN>;
    cudaError_t e = cudaFuncSetAttribute(router_gemm_kernel<BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const dim3 grid((E + kGemmBM - 1) / kGemmBM, (T + BN - 1) / BN, S);
    return launch_kernel(router_gemm_kernel<BN>, grid, dim3(kRouterThreads), C::SMEM, st, false,
                         map_w, map_x, T, H, E, S, out, err);
}

}  // namespace

int router_max_splits(int T, int H, int E) {
    const int ksteps = H / kGemmBK;
    const size_t logits = static_cast<size_t>(T) * E;
    int cap = 1;
    // Powers of two, at least eight K steps per split (fewer, longer splits beat
    // more CTAs: the routing kernel reads every partial sum; measured at decode
    // and prefill against two and four steps), partial sums <= 2^26 floats (256 MB).
    while (cap * 2 <= kRouterMaxSplits && ksteps / (cap * 2) >= 8 &&
           logits * static_cast<size_t>(cap * 2) <= (static_cast<size_t>(1) << 26))
        cap *= 2;
    return cap;
}

RouterPlan router_plan(int T, int H, int E, int num_sms) {
    RouterPlan p;
    p.bn = 16;
    while (p.bn < 256 && p.bn < T) p.bn *= 2;
    const int tiles = ((E + kGemmBM - 1) / kGemmBM) * ((T + p.bn - 1) / p.bn);
    const int ksteps = H / kGemmBK;
    p.splits = 1;
    // Split K while the grid stays within two CTAs per SM, up to
    // router_max_splits (which sizes the workspace).
    const int cap = router_max_splits(T, H, E);
    while (p.splits * 2 <= cap && tiles * p.splits * 2 <= 2 * num_sms) p.splits *= 2;
    return p;
}

cudaError_t launch_router(const RouterPlan& p, const CUtensorMap& map_w, const CUtensorMap& map_x,
                          int T, int H, int E, float* partial, unsigned* err, cudaStream_t st) {
    switch (p.bn) {
        case 16: return launch_router_bn<16>(map_w, map_x, T, H, E, p.splits, partial, err, st);
        case 32: return launch_router_bn<32>(map_w, map_x, T, H, E, p.splits, partial, err, st);
        case 64: return launch_router_bn<64>(map_w, map_x, T, H, E, p.splits, partial, err, st);
        case 128: return launch_router_bn<128>(map_w, map_x, T, H, E, p.splits, partial, err, st);
        case 256: return launch_router_bn<256>(map_w, map_x, T, H, E, p.splits, partial, err, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
