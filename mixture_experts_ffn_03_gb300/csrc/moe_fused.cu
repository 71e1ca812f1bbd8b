// Fused expert phase for decode-sized batches: the gate_up and down grouped
// GEMMs of moe_gemm.cu in one persistent launch, with the same arithmetic
// (the same MMA shapes, the same accumulation order, the same epilogues), so
// its results are bitwise those of the two separate launches.
//
// Aim: with separate launches every SM that runs out of gate_up tiles idles
// until the last gate_up tile anywhere is done (the down grid may start only
// then), and the down pipeline then fills from empty. Here one tile sequence
// holds the gate_up tiles and after them the down tiles; an SM that finishes
// its gate_up work goes straight on to down tiles, whose weights do not
// depend on gate_up at all, and only the h operand of a down tile waits for
// its row tile's gate_up tiles. Measured on GB300 the gain does not
// materialise: the separate launches already overlap through programmatic
// dependent launch, and a down step here uses 20 KB of a 34 KB stage (fewer
// bytes in flight than the down kernel's own ring), so the launch is opt-in
// (moe_set_expert_fusion).
//
// Dependency: a down tile of row tile r reads h over all I features of r, so
// it needs every gate_up tile of r. Each epilogue warp that finishes its part
// of a gate_up tile adds 1 to ready[r] (release, after its h stores); the TMA
// producer of a down tile waits (acquire, bounded in time) until ready[r]
// reaches (gate_up tiles of r) x (epilogue warps) before it loads h. Tiles are
// claimed in index order (all gate_up tiles first) and a CTA never waits on a
// tile it has not yet started, so every awaited gate_up tile is held by a
// resident CTA whose progress does not depend on the waiter; a wait that
// still runs out (e.g. an SM held by someone else's kernel) sets the timeout
// bit in the status word and the CTA leaves, as every wait in these kernels.
//
// Roles (384 threads), as in the separate GEMMs: warp 0 claims tiles and
// issues TMA loads, warp 1 owns TMEM and issues the MMAs, warps 2-3 gather
// hidden rows for gate_up tiles (and pass down stages through), warps 4-11
// drain TMEM. A pipeline stage holds either a gate_up step (128 gate + 128 up
// weight rows and the gathered token rows) or a down step (128 weight rows
// and the tile's h_hi and h_lo rows).
// Sources: "Add Qwen3.5-35B-A3B (support vision and text input)", Description
// (stacked 3D expert weights; per-token sigmoid-gated shared expert).
#include "gemm_common.cuh"
#include "moe_fused.cuh"
#include "routing.cuh"

namespace moe {
namespace {

constexpr int kFusedThreads = 128 + kEpiWarps * 32;
constexpr int kDownBit = 2;  // Tile::shared bit 1 marks a down tile; bit 0 stays "shared expert"

template <int BN>
struct FusedCfg {
    static constexpr int A_BYTES = kGemmBM * kGemmBK * 2;  // 16 KB of weight rows
    static constexpr int B_BYTES = BN * kGemmBK * 2;       // token rows (or one h plane)
    static constexpr int GU_BYTES = 2 * A_BYTES + B_BYTES;
    static constexpr int DN_BYTES = A_BYTES + 2 * B_BYTES;
    static constexpr int STAGE_BYTES = GU_BYTES > DN_BYTES ? GU_BYTES : DN_BYTES;
    static constexpr int CTL_BYTES = 1024;
    static constexpr int EPI_BUFS = 1;  // one y staging buffer per epilogue warp
    static constexpr int EPI_BYTES = kEpiWarps * EPI_BUFS * kStgBytes;
    // gate_up reads its token tile as the MMA's 128-row A operand although
    // only BN rows are loaded: 16 KB - B_BYTES must follow the last stage's
    // token tile (those rows' results are never read).
    static constexpr int TS_SLACK = 16384 - B_BYTES;
    static constexpr int TAIL_BYTES =
        CTL_BYTES + (EPI_BYTES > TS_SLACK - CTL_BYTES ? EPI_BYTES : TS_SLACK - CTL_BYTES);
    static constexpr int STAGES_FIT = (kSmemLimit - 1024 - TAIL_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > kStageCap ? kStageCap : STAGES_FIT;
    static constexpr int A_STAGES = 0;
    static constexpr int CONVERTER_WARPS = 0;
    static constexpr int ACC_COLS = 2 * kGemmBM;  // gate_up: 128 gate + 128 up columns
    static constexpr int ACC_STAGES = 2;
    static constexpr int TMEM_COLS = 512;
    static constexpr int CTL_OFF = STAGES * STAGE_BYTES;
    static constexpr int EPI_OFF = CTL_OFF + CTL_BYTES;
    static constexpr int SMEM = 1024 + CTL_OFF + TAIL_BYTES;
    static_assert(STAGES >= 3, "pipeline depth");
    static_assert(SMEM <= kSmemLimit, "shared memory budget");
    static_assert(STAGE_BYTES % 1024 == 0, "128-byte swizzled tiles start on 1024-byte boundaries");
    static_assert(BN % 16 == 0 && BN <= kFusedMaxBN, "token tile width");
    static_assert(2 * BN <= ACC_COLS, "down accumulator (h_hi and h_lo columns) fits a slot");
};

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_gpu_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Orders this thread's generic-proxy global accesses with its async-proxy
// (TMA) ones.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Wait until *p >= target; false on abort or after the time limit (which
// starts the abort and sets `code`).
__device__ __noinline__ bool wait_ready(const int* p, int target, volatile int* abort_flag,
                                        unsigned* err, unsigned code) {
    if (ld_acquire_gpu(p) >= target) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        __nanosleep(64);
        if (ld_acquire_gpu(p) >= target) return true;
        if ((it & 15u) == 15u) {
            if (*abort_flag) return false;
            if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicOr(err, code);
                return false;
            }
        }
    }
}

// One tile sequence: the gate_up tiles (shared expert's, then routed row
// tiles x feature blocks of I) and after them the down tiles (shared, then
// routed x feature blocks of H), claimed as in TileSched.
template <int BN>
struct FusedSched {
    int nxt, after;
    int4 raw;
    int NG, NT, S_gu, F_gu, F_s, S_dn, F_h;

    __device__ __forceinline__ int4 load(int idx, const GemmArgs& a) const {
        return idx < NG ? load_rowtile(idx, NG, S_gu, F_gu, a)
                        : load_rowtile(idx - NG, NT - NG, S_dn, F_h, a);
    }
    __device__ __forceinline__ Tile make(int idx, int4 r, const GemmArgs& a) const {
        if (idx < NG) return make_tile<BN>(idx, r, NG, S_gu, F_gu, F_s, a);
        Tile ti = make_tile<BN>(idx - NG, r, NT - NG, S_dn, F_h, F_h, a);
        if (ti.n_rows >= 0) ti.shared |= kDownBit;
        return ti;
    }
    __device__ __forceinline__ Tile start(const GemmArgs& a) {
        const int first = blockIdx.x;
        nxt = first < NT ? static_cast<int>(gridDim.x) + atomicAdd(a.sched, 1) : NT;
        return make(first, load(first, a), a);
    }
    __device__ __forceinline__ void prefetch(const GemmArgs& a) {
        raw = load(nxt, a);
        after = nxt < NT ? static_cast<int>(gridDim.x) + atomicAdd(a.sched, 1) : NT;
    }
    __device__ __forceinline__ bool next(Tile& ti, const GemmArgs& a) {
        ti = make(nxt, raw, a);
        nxt = after;
        return true;
    }
};

// Whole-layer launch, before the expert phase: routing of every token (CTA b
// takes tokens b, b + grid, ...) by the CTA's first 256 threads, with the
// routing kernel's arithmetic; the permute by the last CTA to finish
// (completion ticket), in the pipeline's shared memory, which no stage uses
// yet; then every CTA waits (bounded in time) for the permute's flag. Called
// by all threads; false if the wait gave up (the status word then says so).
__device__ __noinline__ bool layer_prologue(uint8_t* smem, const GemmArgs& a, const LayerArgs& l,
                                            volatile int* abort_flag, unsigned code) {
    __shared__ float s_gate[kRouteWarps];
    __shared__ int s_warp[kRouteWarps];
    __shared__ int s_flag;
    const int tid = threadIdx.x;
    if (tid < kSmallThreads)
        for (int t = blockIdx.x; t < a.T; t += gridDim.x)
            route_token_cta<kLayerMaxExperts / 32>(t, a.H, a.E, a.k, l.score_fn, l.logits,
                                                   a.hidden, l.w_g, l.topk_ids, l.topk_w,
                                                   l.gate_logit, l.ids_out, l.w_out, s_gate);
    __threadfence();
    __syncthreads();
    if (tid == 0)
        s_flag = atomicAdd(&l.meta[META_TICKET], 1) == static_cast<int>(gridDim.x) - 1;
    __syncthreads();
    if (s_flag) {
        __threadfence();
        if (tid < kSmallThreads)
            permute_small(a.T, a.E, a.k, l.bn_gu, l.bn_dn, l.topk_ids, l.counts, l.offsets, l.perm,
                          l.inv, l.rt_gu, l.rt_dn, l.meta, l.counts_out,
                          reinterpret_cast<int*>(smem), s_warp);
        __threadfence();
        __syncthreads();
        if (tid == 0) red_release_gpu_add(&l.meta[META_PERMUTED], 1);
    }
    if (tid == 0) s_flag = wait_ready(&l.meta[META_PERMUTED], 1, abort_flag, a.err, code) ? 1 : 0;
    __syncthreads();
    return s_flag != 0;
}

// Whole-layer launch, after the expert phase (and after TMEM is released):
// the CTA counts itself done (its epilogue warps have waited for their y
// stores), waits (bounded) until every CTA is, then combines tokens b, b +
// grid, ... with the combine kernel's arithmetic (over y16 or fp32 rows). No
// combine after an abort.
__device__ __noinline__ void layer_epilogue(const GemmArgs& a, const LayerArgs& l,
                                            volatile int* abort_flag, unsigned code) {
    __shared__ int s_ok;
    const int tid = threadIdx.x;
    if (tid == 0) {
        fence_proxy_async_global();
        __threadfence();
        red_release_gpu_add(&l.meta[META_DONE], 1);
        s_ok = wait_ready(&l.meta[META_DONE], static_cast<int>(gridDim.x), abort_flag, a.err, code)
                   ? 1
                   : 0;
    }
    __syncthreads();
    if (!s_ok) return;
    if (a.yexp) {
        const uint8_t* y = reinterpret_cast<const uint8_t*>(a.y);
        for (int t = blockIdx.x; t < a.T; t += gridDim.x)
            for (int h = tid * 16; h < a.H; h += blockDim.x * 16)
                combine16_y16(t, h, a.T, a.H, a.k, y, l.topk_w, l.inv, l.out);
    } else {
        for (int t = blockIdx.x; t < a.T; t += gridDim.x)
            combine_token(t, a.H, a.k, a.y, a.y + static_cast<size_t>(a.P) * a.H, l.topk_w, l.inv,
                          l.out, tid, blockDim.x);
    }
}

template <int BN, bool LAYER>
__global__ void __launch_bounds__(kFusedThreads, 1)
expert_fused_kernel(const __grid_constant__ GemmMaps gu, const __grid_constant__ GemmMaps dn,
                    const GemmArgs a, int* __restrict__ ready, const LayerArgs l) {
    using C = FusedCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    Ctl* ctl = reinterpret_cast<Ctl*>(smem + C::CTL_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ptx::griddep_launch_dependents();
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&gu.w);
        ptx::prefetch_tmap(&gu.ws);
        ptx::prefetch_tmap(&dn.w);
        ptx::prefetch_tmap(&dn.ws);
        ptx::prefetch_tmap(&dn.h);
        ptx::prefetch_tmap(&dn.hs);
    }
    const uint32_t tmem_base = gemm_setup<C>(ctl, warp, 1 + 2 + kEpiWarps);
    ptx::griddep_wait();  // routing, row tiles and the slot order come from earlier kernels
    volatile int* abort_flag = &ctl->abort;
    const unsigned code = ERR_GATE_UP_TIMEOUT | ERR_DOWN_TIMEOUT;
    bool permuted = true;
    if constexpr (LAYER) permuted = layer_prologue(smem, a, l, abort_flag, code);

    const int R = permuted ? a.meta[META_RT_GU] : 0;
    const int F_gu = (a.I + kGemmBM - 1) / kGemmBM, F_s = (a.I_s + kGemmBM - 1) / kGemmBM;
    const int F_h = (a.H + kGemmBM - 1) / kGemmBM;
    const int RT_s = (a.T + BN - 1) / BN;
    const int tk = a.T * a.k;
    unsigned* err = a.err;

    if (!permuted) {
        // no tile lists: no role runs
    } else if (warp == 0) {
        if (lane == 0) {  // ---------------------------------- tiles + TMA producer
            const uint64_t pol_w = ptx::policy_evict_normal();
            const uint64_t pol_h = ptx::policy_evict_last();  // h rows are re-read per feature block
            int s = 0;
            uint32_t ph = 0, armed = 0, parity_bits = 0;
            bool ok = true;
            FusedSched<BN> sch;
            sch.S_gu = RT_s * F_s;
            sch.F_gu = F_gu;
            sch.F_s = F_s;
            sch.NG = sch.S_gu + R * F_gu;
            sch.S_dn = RT_s * F_h;
            sch.F_h = F_h;
            sch.NT = sch.NG + sch.S_dn + R * F_h;
            Tile ti = sch.start(a);
            int qs = 0;
            uint32_t qph = 0;
            ok = tq_publish(ctl, qs, qph, ti, abort_flag, err, code);
            for (; ok && ti.n_rows >= 0;
                 ok = ok && sch.next(ti, a) && tq_publish(ctl, qs, qph, ti, abort_flag, err, code)) {
                sch.prefetch(a);
                const bool sh = (ti.shared & 1) != 0;
                if (!(ti.shared & kDownBit)) {
                    const CUtensorMap* tm = sh ? &gu.ws : &gu.w;
                    // gate rows f.. of the expert; the map's second plane is the up rows
                    const int row_g = (sh ? 0 : ti.e * 2 * a.I) + ti.f * kGemmBM;
                    for (int ks = 0; ks < a.H / kGemmBK; ++ks) {
                        if (!wait_bar(bar_addr(&ctl->empty[s]), ph ^ 1u, abort_flag, err, code)) {
                            ok = false;
                            break;
                        }
                        const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
                        const uint32_t fb = bar_addr(&ctl->full_a[s]);
                        ptx::mbar_arrive_expect_tx(fb, 2 * C::A_BYTES);
                        ptx::tma_load_3d(sa, tm, fb, ks * kGemmBK, row_g, 0, pol_w);
                        armed |= 1u << s;
                        parity_bits = (parity_bits & ~(1u << s)) | (ph << s);
                        if (++s == C::STAGES) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                } else {
                    // h of this row tile: every gate_up tile of it, every epilogue warp.
                    const int slot = sh ? tk + ti.m0 : ti.p0;
                    const int need = (sh ? F_s : F_gu) * kEpiWarps;
                    if (!wait_ready(ready + slot, need, abort_flag, err, code)) {
                        ok = false;
                        continue;
                    }
                    fence_proxy_async_global();  // h was written with generic stores
                    const int ksteps = (sh ? a.I_s : a.I) / kGemmBK;
                    const CUtensorMap* tw = sh ? &dn.ws : &dn.w;
                    const CUtensorMap* th = sh ? &dn.hs : &dn.h;
                    const int row_w = (sh ? 0 : ti.e * a.H) + ti.f * kGemmBM;
                    for (int ks = 0; ks < ksteps; ++ks) {
                        if (!wait_bar(bar_addr(&ctl->empty[s]), ph ^ 1u, abort_flag, err, code)) {
                            ok = false;
                            break;
                        }
                        const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
                        const uint32_t fb = bar_addr(&ctl->full_a[s]);
                        ptx::mbar_arrive_expect_tx(fb, C::A_BYTES + 2 * C::B_BYTES);
                        ptx::tma_load_2d(sa, tw, fb, ks * kGemmBK, row_w, pol_w);
                        // the tile's h_hi rows, then its h_lo rows (two planes, one request)
                        ptx::tma_load_3d(sa + C::A_BYTES, th, fb, ks * kGemmBK, ti.p0, 0, pol_h);
                        armed |= 1u << s;
                        parity_bits = (parity_bits & ~(1u << s)) | (ph << s);
                        if (++s == C::STAGES) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                }
            }
            if (!ok) drain_tma<C::STAGES>(ctl, armed, parity_bits);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------------------------- MMA issuer
            int s = 0, as = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            int qs = 0;
            uint32_t qph = 0;
            Tile ti;
            while (ok && tq_read(ctl, qs, qph, ti, true, abort_flag, err, code)) {
                const bool down = (ti.shared & kDownBit) != 0;
                const int ksteps =
                    down ? ((ti.shared & 1) ? a.I_s : a.I) / kGemmBK : a.H / kGemmBK;
                // gate_up: tokens on M, 128 gate + 128 up weight rows on N = 256.
                // down: weights on M; h_hi rows (BN) then the tile's h_lo rows on N.
                const uint32_t idesc =
                    down ? ptx::idesc_bf16_f32(kGemmBM, BN + max(16, (ti.n_rows + 15) & ~15))
                         : ptx::idesc_bf16_f32(kGemmBM, 2 * kGemmBM);
                if (!wait_bar(bar_addr(&ctl->tempty[as]), aph ^ 1u, abort_flag, err, code)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + as * C::ACC_COLS;
                for (int ks = 0; ks < ksteps; ++ks) {
                    // full_b completes on every stage use (the gather warps pass
                    // down stages through), which keeps all roles in step.
                    if (!wait_bar(bar_addr(&ctl->full_a[s]), ph, abort_flag, err, code) ||
                        !wait_bar(bar_addr(&ctl->full_b[s]), ph, abort_flag, err, code)) {
                        ok = false;
                        break;
                    }
                    ptx::fence_proxy_async_smem();  // gathered rows were written by cp.async
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
                    const uint64_t dw = ptx::smem_desc_sw128(sa);
                    if (!down) {
                        const uint64_t dx = ptx::smem_desc_sw128(sa + 2 * C::A_BYTES);
#pragma unroll
                        for (int kk = 0; kk < kGemmBK / 16; ++kk)
                            ptx::mma_bf16_ss(d, dx + 2 * kk, dw + 2 * kk, idesc,
                                             (ks | kk) != 0 ? 1u : 0u);
                    } else {
                        const uint64_t dh = ptx::smem_desc_sw128(sa + C::A_BYTES);
#pragma unroll
                        for (int kk = 0; kk < kGemmBK / 16; ++kk)
                            ptx::mma_bf16_ss(d, dw + 2 * kk, dh + 2 * kk, idesc,
                                             (ks | kk) != 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(bar_addr(&ctl->empty[s]));
                    if (++s == C::STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(bar_addr(&ctl->tfull[as]));
                if (++as == C::ACC_STAGES) {
                    as = 0;
                    aph ^= 1u;
                }
            }
            if (!ok) {
                ptx::mma_commit(bar_addr(&ctl->drain));
                wait_bounded(bar_addr(&ctl->drain), 0);
            }
        }
    } else if (warp < 4) {  // ------------------------------ row gather (64 threads)
        // Thread gl copies 16-byte chunk c of rows r_first, r_first + 8, ...;
        // with the 128-byte swizzle that chunk lands at position c ^ r_first.
        constexpr int RPT = BN / 8;
        const int gl = (warp - 2) * 32 + lane;
        const int c = gl & 7;
        const int r_first = gl >> 3;
        const uint32_t swz = static_cast<uint32_t>((c ^ r_first) << 4);
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        int qs = 0;
        uint32_t qph = 0;
        Tile ti;
        while (ok && tq_read(ctl, qs, qph, ti, false, abort_flag, err, code)) {
            if (ti.shared & kDownBit) {
                const int ksteps = ((ti.shared & 1) ? a.I_s : a.I) / kGemmBK;
                for (int ks = 0; ks < ksteps; ++ks) {
                    if (!wait_bar(bar_addr(&ctl->empty[s]), ph ^ 1u, abort_flag, err, code)) {
                        ok = false;
                        break;
                    }
                    ptx::mbar_arrive(bar_addr(&ctl->full_b[s]));
                    if (++s == C::STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                continue;
            }
            uint32_t trow[RPT];  // token (hidden row) of each row this thread copies
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                const int r = r_first + 8 * j;
                uint32_t t = 0;
                if (r < ti.n_rows) t = (ti.shared & 1) ? ti.m0 + r : a.perm[ti.p0 + r] / a.k;
                trow[j] = t;
            }
            const __nv_bfloat16* col = a.hidden + c * 8;
            for (int ks = 0; ks < a.H / kGemmBK; ++ks) {
                if (!wait_bar(bar_addr(&ctl->empty[s]), ph ^ 1u, abort_flag, err, code)) {
                    ok = false;
                    break;
                }
                const uint32_t sb = ptx::smem_u32(smem + s * C::STAGE_BYTES + 2 * C::A_BYTES);
                const __nv_bfloat16* src = col + ks * kGemmBK;
#pragma unroll
                for (int j = 0; j < RPT; ++j) {
                    const int r = r_first + 8 * j;
                    if (r < ti.n_rows)
                        ptx::cp_async_16(sb + r * 128 + swz, src + static_cast<size_t>(trow[j]) * a.H);
                }
                ptx::cp_async_arrive_noinc(bar_addr(&ctl->full_b[s]));
                if (++s == C::STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        ptx::cp_async_wait_all();
    } else {  // ------------------------------------------- epilogue (warps 4-11)
        const int we = warp - 4, q = warp & 3, half = we >> 2;
        uint8_t* stg = smem + C::EPI_OFF + we * C::EPI_BUFS * kStgBytes;
        uint32_t nbuf = 0;
        int as = 0;
        uint32_t aph = 0;
        int qs = 0;
        uint32_t qph = 0;
        Tile ti;
        while (tq_read(ctl, qs, qph, ti, false, abort_flag, err, code)) {
            if (!wait_bar(bar_addr(&ctl->tfull[as]), aph, abort_flag, err, code)) break;
            ptx::tc_fence_after();
            const uint32_t slot = tmem_base + as * C::ACC_COLS;
            if (!(ti.shared & kDownBit)) {  // the same epilogues as the separate kernels
                gate_up_ts_epilogue_tile(ti, slot, q, half, lane, a);
                // This warp's share of the tile's h is written: make it visible
                // to the TMA loads of other CTAs, then count it for the row tile.
                fence_proxy_async_global();
                __threadfence();
                __syncwarp();
                if (lane == 0)
                    red_release_gpu_add(ready + ((ti.shared & 1) ? tk + ti.m0 : ti.p0), 1);
            } else {
                down_epilogue_tile<BN, C::EPI_BUFS>(ti, slot, q, half, lane, stg, nbuf, &dn.st[0],
                                                    a);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_addr(&ctl->tempty[as]));
            if (++as == C::ACC_STAGES) {
                as = 0;
                aph ^= 1u;
            }
        }
        if (lane == 0) {
            ptx::bulk_wait_all();
            if constexpr (LAYER) fence_proxy_async_global();  // y is read by other CTAs next
        }
    }
    gemm_teardown<C>(tmem_base, warp);
    if constexpr (LAYER) layer_epilogue(a, l, abort_flag, code);
}

template <int BN>
cudaError_t launch_fused_bn(const GemmMaps& gu, const GemmMaps& dn, const GemmArgs& a, int* ready,
                            int max_tiles, int num_sms, cudaStream_t st) {
    using C = FusedCfg<BN>;
    cudaError_t e = cudaFuncSetAttribute(expert_fused_kernel<BN, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const int grid = max_tiles < num_sms ? max_tiles : num_sms;
    if (grid <= 0) return cudaSuccess;
    return launch_kernel(expert_fused_kernel<BN, false>, dim3(grid), dim3(kFusedThreads), C::SMEM,
                         st, true, gu, dn, a, ready, LayerArgs{});
}

// One CTA per SM: every CTA routes, waits for the permute, takes expert
// tiles (or none) and combines. Its CTAs wait on one another (the permute
// flag, the done count), so the launch is cooperative: all of them resident.
template <int BN>
cudaError_t launch_layer_bn(const GemmMaps& gu, const GemmMaps& dn, const GemmArgs& a, int* ready,
                            const LayerArgs& l, int num_sms, cudaStream_t st) {
    using C = FusedCfg<BN>;
    cudaError_t e = cudaFuncSetAttribute(expert_fused_kernel<BN, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    return launch_kernel_cooperative(expert_fused_kernel<BN, true>, dim3(num_sms),
                                     dim3(kFusedThreads), C::SMEM, st, gu, dn, a, ready, l);
}

}  // namespace

cudaError_t launch_expert_fused(int bn, const GemmMaps& gu, const GemmMaps& dn, const GemmArgs& a,
                                int* ready, int max_tiles, int num_sms, cudaStream_t st) {
    switch (bn) {
        case 16: return launch_fused_bn<16>(gu, dn, a, ready, max_tiles, num_sms, st);
        case 32: return launch_fused_bn<32>(gu, dn, a, ready, max_tiles, num_sms, st);
        case 64: return launch_fused_bn<64>(gu, dn, a, ready, max_tiles, num_sms, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_layer_fused(int bn, const GemmMaps& gu, const GemmMaps& dn, const GemmArgs& a,
                               int* ready, const LayerArgs& l, int num_sms, cudaStream_t st) {
    switch (bn) {
        case 16: return launch_layer_bn<16>(gu, dn, a, ready, l, num_sms, st);
        case 32: return launch_layer_bn<32>(gu, dn, a, ready, l, num_sms, st);
        case 64: return launch_layer_bn<64>(gu, dn, a, ready, l, num_sms, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
