// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA, persistent and warp-specialised.
//
// Tiles come from a device-built list of row tiles {expert, first row, rows,
// first sorted position}, so empty experts cost nothing and no host
// synchronisation is needed; the shared expert's tiles come first in the
// list. Each GEMM puts the operand with 128 useful rows on the MMA's M side
// (one TMEM lane per row) and the other on N; which one depends on the tile
// width BN (tokens per tile):
//
// gate_up, BN <= 128: tokens on M (rows past the tile's end unused), NF gate
//   rows then NF up rows of the expert on N (NF = 64 for BN <= 32, else 128),
//   one MMA per K step, two accumulator stages; a thread owns one token in
//   the epilogue. BN = 160 / 256: weights on M (128 gate rows, 128 up rows:
//   two MMAs sharing the B operand X, the gathered hidden rows), one
//   accumulator stage.
//   The epilogue writes h = silu(G) * U as a bf16 high/low pair (h_hi =
//   bf16(h), h_lo = bf16(h - h_hi)).
// down, BN <= 32: weights on M (128 output features); the tile's h_hi and
//   h_lo rows are adjacent in shared memory and form the N side of one MMA
//   against the same weight tile; two 64-K chunks per pipeline stage; the
//   epilogue adds the two column blocks and writes y rows per (token, slot)
//   (fp32, or y16 codes where fp32 y would be large). BN = 64
//   (down_stk_kernel): the tile's h_hi rows stacked over its h_lo rows on M,
//   256 output features on N, the two halves added in the epilogue. BN = 128
//   (down_ts_kernel): tokens on M, 256 output features on N, h_hi and h_lo as
//   two A operands into one accumulator; y as y16 codes (16 bits per value
//   and one exponent byte per 32 values). The shared expert's rows are scaled
//   by the per-token gate sigmoid(x . w_g).
// Sources: "Add Qwen3.5-35B-A3B (support vision and text input)", Description
// (stacked 3D expert weights; per-token sigmoid-gated shared expert); the
// SwiGLU expert FFN is the plain reading of the stacked gate/up layout.
//
// Warp roles (384 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues the MMAs, warps 2-3 gather hidden rows with cp.async (gate_up only),
// warps 4-11 drain TMEM in the epilogue (warp w reads TMEM lanes
// 32*(w%4)..; two warps per lane quadrant split the columns) and write
// results with 16-byte stores (h) or TMA box stores through shared memory (y).
// Every wait on a pipeline barrier gives up after a time limit, sets an error
// bit in the workspace status word and lets the CTA finish cleanly.
#include "gemm_common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128 + kEpiWarps * 32;     // TMA, MMA, 2 gather warps, epilogue

template <int BN, bool GU>
struct Cfg {
    // gate_up with BN <= 128 puts the tokens on the MMA's M side (M = 128) and
    // the 128 gate + 128 up weight rows on N = 256: one MMA per K slice.
    // gate_up with BN = 256 and down keep the weights on M.
    static constexpr bool TS = GU && BN <= 128;
    // Weight rows per tile and operand: 128 output features, or for the
    // tokens-on-M gate_up NF gate and NF up rows.
    static constexpr int NF = TS ? gate_up_ts_features(BN) : kGemmBM;
    static constexpr int A_BYTES = NF * kGemmBK * 2;       // 16 KB weight tile (8 KB at NF = 64)
    static constexpr int B_BYTES = BN * kGemmBK * 2;       // token tile
    // down: a stage holds KC consecutive 64-K chunks, loaded as one weight
    // request ([chunk][128 rows]) and one h request ([chunk][h_hi, h_lo][BN
    // rows]): at decode widths the h tile is small, and two requests per 20 KB
    // left the TMA request rate, not HBM, setting the pace.
    static constexpr int KC = GU ? 1 : kDownChunks;
    static constexpr int STAGE_BYTES = GU ? (2 * A_BYTES + B_BYTES) : KC * (A_BYTES + 2 * B_BYTES);
    static constexpr int CTL_BYTES = 1024;
    // Store staging: gate_up stages each chunk in one buffer per epilogue warp
    // and writes it with plain stores; down uses TMA stores from two buffers
    // per warp, or one when that buys the pipeline another stage.
    static constexpr int STAGES_2BUF =
        (kSmemLimit - 1024 - CTL_BYTES - kEpiWarps * 2 * kStgBytes) / STAGE_BYTES;
    static constexpr int STAGES_1BUF =
        (kSmemLimit - 1024 - CTL_BYTES - kEpiWarps * kStgBytes) / STAGE_BYTES;
    static constexpr int EPI_BUFS =
        (GU || (STAGES_1BUF > STAGES_2BUF && STAGES_2BUF < kStageCap)) ? 1 : 2;
    static constexpr int EPI_BYTES = TS ? 0 : kEpiWarps * EPI_BUFS * kStgBytes;
    // TS: the MMA reads the token tile as 128 rows although only BN are loaded
    // (results of the extra rows are never used), so 16 KB - B_BYTES of
    // shared memory must follow the last stage's token tile.
    static constexpr int TS_SLACK = TS ? 16384 - B_BYTES : 0;
    static constexpr int TAIL_BYTES =
        CTL_BYTES + (EPI_BYTES > TS_SLACK - CTL_BYTES ? EPI_BYTES : TS_SLACK - CTL_BYTES);
    static constexpr int STAGES_FIT = (kSmemLimit - 1024 - TAIL_BYTES) / STAGE_BYTES;
    // the 64-feature gate_up steps are half as large: let them keep as many
    // bytes in flight as the others
    static constexpr int STAGE_CAP = NF < kGemmBM ? kMaxStages : kStageCap;
    static constexpr int STAGES = STAGES_FIT > STAGE_CAP ? STAGE_CAP : STAGES_FIT;
    static constexpr int A_STAGES = 0;                  // no TMEM weight stages
    static constexpr int CONVERTER_WARPS = 0;
    static constexpr int ACC_COLS = TS ? 2 * NF : 2 * BN;  // TMEM columns per accumulator set
    static constexpr int ACC_STAGES = (2 * ACC_COLS <= 512) ? 2 : 1;
    static constexpr int TMEM_USED = ACC_COLS * ACC_STAGES;
    static constexpr int TMEM_COLS = TMEM_USED <= 32    ? 32
                                     : TMEM_USED <= 64  ? 64
                                     : TMEM_USED <= 128 ? 128
                                     : TMEM_USED <= 256 ? 256
                                                        : 512;
    static constexpr int CTL_OFF = STAGES * STAGE_BYTES;
    static constexpr int EPI_OFF = CTL_OFF + CTL_BYTES;
    static constexpr int SMEM = 1024 + CTL_OFF + TAIL_BYTES;
    static_assert(STAGES >= 2, "pipeline needs two stages");
    static_assert(SMEM <= kSmemLimit, "shared memory budget");
    static_assert(BN % 16 == 0 && BN <= 256, "MMA N");
    static_assert(BN % 8 == 0, "row gather: 8 rows per pass");
    static_assert(GU || BN <= 128, "down: h_hi and h_lo rows share one MMA of N <= 256");
    static_assert(A_BYTES % 1024 == 0 && (2 * B_BYTES) % 1024 == 0, "chunks keep the swizzle phase");
};

// ================================================================ gate_up
template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
gate_up_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs a) {
    using C = Cfg<BN, true>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    Ctl* ctl = reinterpret_cast<Ctl*>(smem + C::CTL_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ptx::griddep_launch_dependents();
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&maps.w);
        ptx::prefetch_tmap(&maps.ws);
    }
    const uint32_t tmem_base = gemm_setup<C>(ctl, warp, 1 + 2 + kEpiWarps);
    const int F = (a.I + C::NF - 1) / C::NF, F_s = (a.I_s + C::NF - 1) / C::NF;
    if (warp == 0 && lane == 0 && a.w_gu != nullptr) {
        // While routing finishes, HBM is idle: prefetch into L2 the gate and up
        // rows of routed tile blockIdx.x as it would be if every expert had a
        // row tile (expert blockIdx.x / F, feature block blockIdx.x % F). Tiles
        // are claimed in expert order, so the first wave reads about these.
        const int e = static_cast<int>(blockIdx.x) / F, f = static_cast<int>(blockIdx.x) % F;
        if (e < a.E) {
            // this tile's gate rows (and as many up rows); never past the expert
            const int rows = min(C::NF, a.I - f * C::NF);
            const size_t plane = static_cast<size_t>(rows) * a.H * 2;
            const uint8_t* g = reinterpret_cast<const uint8_t*>(a.w_gu) +
                               (static_cast<size_t>(e) * 2 * a.I + static_cast<size_t>(f) * C::NF) *
                                   a.H * 2;
            const uint8_t* u = g + static_cast<size_t>(a.I) * a.H * 2;
            constexpr uint32_t kChunk = 64 * 1024;
            for (size_t o = 0; o < plane; o += kChunk) {
                const uint32_t n = static_cast<uint32_t>(plane - o < kChunk ? plane - o : kChunk);
                ptx::prefetch_l2_bulk(g + o, n);
                ptx::prefetch_l2_bulk(u + o, n);
            }
        }
    }
    ptx::griddep_wait();  // routing, tile lists and the slot order come from earlier kernels

    const int R = a.meta[META_RT_GU];
    const int shared_tiles = ((a.T + BN - 1) / BN) * F_s;
    const int num_tiles = R * F + shared_tiles;
    const int ksteps = a.H / kGemmBK;
    volatile int* abort_flag = &ctl->abort;
    unsigned* err = a.err;
    const unsigned code = ERR_GATE_UP_TIMEOUT;

    if (warp == 0) {
        if (lane == 0) {  // ---------------------------------- TMA producer
            // Each weight tile is read by one tile (decode, prefill, wide) or by the
            // few row tiles of a hot expert, which run at about the same time:
            // evict it first, so that the hidden rows, read k times, stay in L2.
            const uint64_t pol = ptx::policy_evict_first();
            int s = 0;
            uint32_t ph = 0, armed = 0, parity_bits = 0;
            bool ok = true;
            TileSched<BN> sch;
            Tile ti = sch.start(num_tiles, shared_tiles, F, F_s, a);
            int qs = 0;
            uint32_t qph = 0;
            ok = tq_publish(ctl, qs, qph, ti, abort_flag, err, code);
            for (; ok && ti.n_rows >= 0;
                 ok = ok && sch.next(ti, a) && tq_publish(ctl, qs, qph, ti, abort_flag, err, code)) {
                sch.prefetch(a);
                const CUtensorMap* tm = ti.shared ? &maps.ws : &maps.w;
                // gate rows f.. of the expert; the map's second plane is the up rows
                const int row_g = (ti.shared ? 0 : ti.e * 2 * a.I) + ti.f * C::NF;
                for (int ks = 0; ks < ksteps; ++ks) {
                    if (!wait_bar(bar_addr(&ctl->empty[s]), ph ^ 1u, abort_flag, err, code)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
                    const uint32_t fb = bar_addr(&ctl->full_a[s]);
                    ptx::mbar_arrive_expect_tx(fb, 2 * C::A_BYTES);
                    ptx::tma_load_3d(sa, tm, fb, ks * kGemmBK, row_g, 0, pol);  // gate, then up
                    armed |= 1u << s;
                    parity_bits = (parity_bits & ~(1u << s)) | (ph << s);
                    if (++s == C::STAGES) {
                        s = 0;
                        ph ^= 1u;
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
                const int n_mma = max(16, (ti.n_rows + 15) & ~15);
                const uint32_t idesc = C::TS ? ptx::idesc_bf16_f32(kGemmBM, 2 * C::NF)
                                             : ptx::idesc_bf16_f32(kGemmBM, n_mma);
                if (!wait_bar(bar_addr(&ctl->tempty[as]), aph ^ 1u, abort_flag, err, code)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_gate = tmem_base + as * C::ACC_COLS;
                const uint32_t d_up = d_gate + BN;
                for (int ks = 0; ks < ksteps; ++ks) {
                    if (!wait_bar(bar_addr(&ctl->full_a[s]), ph, abort_flag, err, code) ||
                        !wait_bar(bar_addr(&ctl->full_b[s]), ph, abort_flag, err, code)) {
                        ok = false;
                        break;
                    }
                    ptx::fence_proxy_async_smem();  // gathered rows were written by cp.async
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
                    const uint64_t da0 = ptx::smem_desc_sw128(sa);
                    const uint64_t da1 = ptx::smem_desc_sw128(sa + C::A_BYTES);
                    const uint64_t db = ptx::smem_desc_sw128(sa + 2 * C::A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < kGemmBK / 16; ++kk) {
                        const uint32_t acc = (ks | kk) != 0 ? 1u : 0u;
                        // +32 bytes of K per step, in 16-byte descriptor units
                        if constexpr (C::TS) {
                            // D[token, 0:128] = gate, D[token, 128:256] = up: the gate
                            // and up boxes are adjacent, one descriptor spans both.
                            ptx::mma_bf16_ss(d_gate, db + 2 * kk, da0 + 2 * kk, idesc, acc);
                        } else {
                            ptx::mma_bf16_ss(d_gate, da0 + 2 * kk, db + 2 * kk, idesc, acc);
                            ptx::mma_bf16_ss(d_up, da1 + 2 * kk, db + 2 * kk, idesc, acc);
                        }
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
        constexpr int RPT = BN / 8;  // rows per thread at most
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
            // source row of each row this thread copies: a token's hidden row, or a
            // pre-gathered row (expert parallelism)
            const bool pre = !ti.shared && a.xrows != nullptr;
            uint32_t trow[RPT];
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                const int r = r_first + 8 * j;
                uint32_t t = 0;
                if (r < ti.n_rows)
                    t = ti.shared ? ti.m0 + r : (pre ? ti.p0 + r : a.perm[ti.p0 + r] / a.k);
                trow[j] = t;
            }
            const __nv_bfloat16* col = (pre ? a.xrows : a.hidden) + c * 8;
            // Each hidden row is gathered by the k experts of its token: keep it
            // in L2. The 256-byte L2 prefetch also brings in the row's next K step.
            const uint64_t pol_x = ptx::policy_evict_last();
            for (int ks = 0; ks < ksteps; ++ks) {
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
                        ptx::cp_async_16_hint(sb + r * 128 + swz,
                                              src + static_cast<size_t>(trow[j]) * a.H, pol_x);
                }
                ptx::cp_async_arrive_noinc(bar_addr(&ctl->full_b[s]));
                if (++s == C::STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        ptx::cp_async_wait_all();
    } else if constexpr (C::TS) {  // ------------------------- epilogue (warps 4-11)
        // Tokens on TMEM lanes: gate_up_ts_epilogue_tile per tile.
        const int we = warp - 4, q = warp & 3, half = we >> 2;
        int as = 0;
        uint32_t aph = 0;
        int qs = 0;
        uint32_t qph = 0;
        Tile ti;
        while (tq_read(ctl, qs, qph, ti, false, abort_flag, err, code)) {
            if (!wait_bar(bar_addr(&ctl->tfull[as]), aph, abort_flag, err, code)) break;
            ptx::tc_fence_after();
            gate_up_ts_epilogue_tile<C::NF>(ti, tmem_base + as * C::ACC_COLS, q, half, lane, a);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_addr(&ctl->tempty[as]));
            if (++as == C::ACC_STAGES) {
                as = 0;
                aph ^= 1u;
            }
        }
    } else {  // ------------------------------------------- epilogue (warps 4-11)
        // Warp we drains TMEM lanes 32*(warp % 4).. (32 intermediate features)
        // for the 16-column chunks 16*(we / 4) + 32*j of each tile. Each chunk
        // is transposed through the warp's own shared buffer (token rows of 32
        // features, 64 bytes each) and written with 16-byte stores, four lanes
        // per row: no store waits on an earlier one, so the accumulator is
        // released as soon as the last chunk has been read out of TMEM.
        const int we = warp - 4, q = warp & 3, half = we >> 2;
        __nv_bfloat16* shi = reinterpret_cast<__nv_bfloat16*>(smem + C::EPI_OFF + we * kStgBytes);
        __nv_bfloat16* slo = shi + kEpiRows * kEpiCols;
        int as = 0;
        uint32_t aph = 0;
        int qs = 0;
        uint32_t qph = 0;
        Tile ti;
        while (tq_read(ctl, qs, qph, ti, false, abort_flag, err, code)) {
            if (!wait_bar(bar_addr(&ctl->tfull[as]), aph, abort_flag, err, code)) break;
            ptx::tc_fence_after();
            const int n_feat = ti.shared ? a.I_s : a.I;
            const int i0 = ti.f * kGemmBM + q * kEpiCols;  // feature of lane 0
            const bool warp_valid = i0 < n_feat;            // I, I_s are multiples of 64
            __nv_bfloat16* dhi = ti.shared ? a.hs_hi : a.h_hi;
            __nv_bfloat16* dlo = ti.shared ? a.hs_lo : a.h_lo;
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + as * C::ACC_COLS;
            for (int c0 = half * kEpiRows; c0 < ti.n_rows; c0 += 2 * kEpiRows) {
                uint32_t g[kEpiRows], u[kEpiRows];
                ptx::tmem_ld_32x32b_x16(tb + c0, g);
                ptx::tmem_ld_32x32b_x16(tb + BN + c0, u);
                ptx::tmem_ld_wait();
                if (!warp_valid) continue;
                const int rows = min(kEpiRows, ti.n_rows - c0);
                __syncwarp();  // the previous chunk's rows have been read back
#pragma unroll
                for (int n = 0; n < kEpiRows; ++n) {
                    const float gv = __uint_as_float(g[n]);
                    const float h = __fdividef(gv, 1.f + __expf(-gv)) * __uint_as_float(u[n]);
                    const __nv_bfloat16 hi = __float2bfloat16_rn(h);
                    shi[n * kEpiCols + lane] = hi;
                    slo[n * kEpiCols + lane] = __float2bfloat16_rn(h - __bfloat162float(hi));
                }
                __syncwarp();
                // 16 rows x 64 bytes per plane: lane l moves 16-byte pieces l and l + 32
                // (row v / 4, features 8 (v % 4) ..) of both planes.
#pragma unroll
                for (int v = lane; v < kEpiRows * 4; v += 32) {
                    const int r = v >> 2, part = v & 3;
                    if (r < rows) {
                        const size_t o = static_cast<size_t>(ti.p0 + c0 + r) * n_feat + i0 + part * 8;
                        *reinterpret_cast<uint4*>(dhi + o) = reinterpret_cast<const uint4*>(shi)[v];
                        *reinterpret_cast<uint4*>(dlo + o) = reinterpret_cast<const uint4*>(slo)[v];
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_addr(&ctl->tempty[as]));
            if (++as == C::ACC_STAGES) {
                as = 0;
                aph ^= 1u;
            }
        }
    }
    gemm_teardown<C>(tmem_base, warp);
}

// =================================================================== down
template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
down_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs a) {
    using C = Cfg<BN, false>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    Ctl* ctl = reinterpret_cast<Ctl*>(smem + C::CTL_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ptx::griddep_launch_dependents();
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&maps.w);
        ptx::prefetch_tmap(&maps.ws);
        ptx::prefetch_tmap(&maps.h);
        ptx::prefetch_tmap(&maps.hs);
    }
    const uint32_t tmem_base = gemm_setup<C>(ctl, warp, 1 + kEpiWarps);
    ptx::griddep_wait();  // h, tile lists and the gate logits come from earlier kernels

    const int R = a.meta[META_RT_DN];
    const int F = (a.H + kGemmBM - 1) / kGemmBM;
    const int shared_tiles = ((a.T + BN - 1) / BN) * F;
    const int num_tiles = R * F + shared_tiles;
    volatile int* abort_flag = &ctl->abort;
    unsigned* err = a.err;
    const unsigned code = ERR_DOWN_TIMEOUT;

    if (warp == 0) {
        if (lane == 0) {  // ---------------------------------- TMA producer
            const uint64_t pol_w = ptx::policy_evict_normal();
            const uint64_t pol_h = ptx::policy_evict_last();  // h rows are re-read per feature block
            int s = 0;
            uint32_t ph = 0, armed = 0, parity_bits = 0;
            bool ok = true;
            TileSched<BN> sch;
            Tile ti = sch.start(num_tiles, shared_tiles, F, F, a);
            int qs = 0;
            uint32_t qph = 0;
            ok = tq_publish(ctl, qs, qph, ti, abort_flag, err, code);
            for (; ok && ti.n_rows >= 0;
                 ok = ok && sch.next(ti, a) && tq_publish(ctl, qs, qph, ti, abort_flag, err, code)) {
                sch.prefetch(a);
                const int ksteps = ((ti.shared ? a.I_s : a.I) / kGemmBK + C::KC - 1) / C::KC;
                const CUtensorMap* tw = ti.shared ? &maps.ws : &maps.w;
                const CUtensorMap* th = ti.shared ? &maps.hs : &maps.h;
                const int row_w = (ti.shared ? 0 : ti.e * a.H) + ti.f * kGemmBM;
                for (int ks = 0; ks < ksteps; ++ks) {
                    if (!wait_bar(bar_addr(&ctl->empty[s]), ph ^ 1u, abort_flag, err, code)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
                    const uint32_t fb = bar_addr(&ctl->full_a[s]);
                    ptx::mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
                    // KC chunks of 128 weight rows; then per chunk the tile's h_hi
                    // rows and its h_lo rows (chunks past K read as zeros)
                    ptx::tma_load_3d(sa, tw, fb, 0, row_w, ks * C::KC, pol_w);
                    ptx::tma_load_4d(sa + C::KC * C::A_BYTES, th, fb, 0, ti.p0, 0, ks * C::KC, pol_h);
                    armed |= 1u << s;
                    parity_bits = (parity_bits & ~(1u << s)) | (ph << s);
                    if (++s == C::STAGES) {
                        s = 0;
                        ph ^= 1u;
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
                const int ksteps = ((ti.shared ? a.I_s : a.I) / kGemmBK + C::KC - 1) / C::KC;
                // h_lo rows sit right after the BN h_hi rows in shared memory, so
                // one MMA of N = BN + rows covers both halves: accumulator
                // columns [0, BN) hold W h_hi, columns [BN, BN + rows) W h_lo.
                const int n_mma = BN + max(16, (ti.n_rows + 15) & ~15);
                const uint32_t idesc = ptx::idesc_bf16_f32(kGemmBM, n_mma);
                if (!wait_bar(bar_addr(&ctl->tempty[as]), aph ^ 1u, abort_flag, err, code)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + as * C::ACC_COLS;
                for (int ks = 0; ks < ksteps; ++ks) {
                    if (!wait_bar(bar_addr(&ctl->full_a[s]), ph, abort_flag, err, code)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
#pragma unroll
                    for (int c = 0; c < C::KC; ++c) {
                        const uint64_t da = ptx::smem_desc_sw128(sa + c * C::A_BYTES);
                        const uint64_t dh =
                            ptx::smem_desc_sw128(sa + C::KC * C::A_BYTES + c * 2 * C::B_BYTES);
#pragma unroll
                        for (int kk = 0; kk < kGemmBK / 16; ++kk) {
                            const uint32_t acc = (ks | c | kk) != 0 ? 1u : 0u;
                            ptx::mma_bf16_ss(d, da + 2 * kk, dh + 2 * kk, idesc, acc);
                        }
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
    } else if (warp >= 4) {  // ------------------------------ epilogue (warps 4-11)
        down_epilogue<C, BN>(smem, ctl, tmem_base, warp, lane, &maps.st[0], a, abort_flag, err,
                             code);
    }
    gemm_teardown<C>(tmem_base, warp);
}

// ====================================================== down, tokens on M
// Tiles of up to 128 tokens of one expert against 256 output features:
// D[token, 0:N] = h_hi W^T + h_lo W^T, where the h_hi and h_lo tiles are two A
// operands (M = 128 token rows) accumulating into one TMEM accumulator and the
// weight tile (N = 256 rows of W_down[e]) is the B operand. Each h row is read
// once per 256 output features (twice as few as with the weights on M) and the
// epilogue drains a single accumulator. Used when groups are large enough to
// fill most of the 128 token rows.
struct DownTs {
    static constexpr int BM = 128;                          // token rows per tile (MMA M)
    static constexpr int NF = 256;                          // output features per tile (MMA N)
    static constexpr int A_BYTES = BM * kGemmBK * 2;        // 16 KB: h_hi or h_lo tile
    static constexpr int W_BYTES = NF * kGemmBK * 2;        // 32 KB: weight tile (two boxes)
    static constexpr int STAGE_BYTES = 2 * A_BYTES + W_BYTES;
    static constexpr int STG_BYTES = 32 * 32 * 4;           // one warp's store box (32 rows x 64 B used)
    static constexpr int EPI_BYTES = kEpiWarps * STG_BYTES;
    static constexpr int CTL_BYTES = 1024;
    static constexpr int STAGES_FIT = (kSmemLimit - 1024 - EPI_BYTES - CTL_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > kStageCap ? kStageCap : STAGES_FIT;
    static constexpr int EPI_OFF = STAGES * STAGE_BYTES;    // 1024-byte aligned (swizzled boxes)
    static constexpr int CTL_OFF = EPI_OFF + EPI_BYTES;
    static constexpr int SMEM = 1024 + CTL_OFF + CTL_BYTES;
    static constexpr int ACC_COLS = NF;
    static constexpr int A_STAGES = 0;
    static constexpr int CONVERTER_WARPS = 0;
    static constexpr int ACC_STAGES = 2;
    static constexpr int TMEM_COLS = 512;
    static_assert(STAGES >= 2, "pipeline needs two stages");
    static_assert(SMEM <= kSmemLimit, "shared memory budget");
    static_assert(EPI_OFF % 1024 == 0 && STG_BYTES % 1024 == 0, "swizzled staging alignment");
};

__global__ void __launch_bounds__(kThreads, 1)
down_ts_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs a) {
    using C = DownTs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    Ctl* ctl = reinterpret_cast<Ctl*>(smem + C::CTL_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ptx::griddep_launch_dependents();
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&maps.w);
        ptx::prefetch_tmap(&maps.ws);
        ptx::prefetch_tmap(&maps.h);
        ptx::prefetch_tmap(&maps.hs);
        ptx::prefetch_tmap(&maps.st[1]);
    }
    const uint32_t tmem_base = gemm_setup<C>(ctl, warp, 1 + kEpiWarps);
    ptx::griddep_wait();  // h, tile lists and the gate logits come from earlier kernels

    const int R = a.meta[META_RT_DN];
    const int F = (a.H + C::NF - 1) / C::NF;
    const int shared_tiles = ((a.T + C::BM - 1) / C::BM) * F;
    const int num_tiles = R * F + shared_tiles;
    volatile int* abort_flag = &ctl->abort;
    unsigned* err = a.err;
    const unsigned code = ERR_DOWN_TIMEOUT;

    if (warp == 0) {
        if (lane == 0) {  // ---------------------------------- TMA producer
            const uint64_t pol_w = ptx::policy_evict_normal();
            const uint64_t pol_h = ptx::policy_evict_last();  // h rows are re-read per feature block
            int s = 0;
            uint32_t ph = 0, armed = 0, parity_bits = 0;
            bool ok = true;
            TileSched<C::BM> sch;
            Tile ti = sch.start(num_tiles, shared_tiles, F, F, a);
            int qs = 0;
            uint32_t qph = 0;
            ok = tq_publish(ctl, qs, qph, ti, abort_flag, err, code);
            for (; ok && ti.n_rows >= 0;
                 ok = ok && sch.next(ti, a) && tq_publish(ctl, qs, qph, ti, abort_flag, err, code)) {
                sch.prefetch(a);
                const int ksteps = (ti.shared ? a.I_s : a.I) / kGemmBK;
                const CUtensorMap* tw = ti.shared ? &maps.ws : &maps.w;
                const CUtensorMap* th = ti.shared ? &maps.hs : &maps.h;
                // Rows past this expert's H (a ragged last block) read the next
                // expert's rows or zero fill; their columns are never stored.
                const int row_w = (ti.shared ? 0 : ti.e * a.H) + ti.f * C::NF;
                for (int ks = 0; ks < ksteps; ++ks) {
                    if (!wait_bar(bar_addr(&ctl->empty[s]), ph ^ 1u, abort_flag, err, code)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
                    const uint32_t fb = bar_addr(&ctl->full_a[s]);
                    ptx::mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
                    // h_hi then h_lo tile (one request), then 256 weight rows (one request)
                    ptx::tma_load_3d(sa, th, fb, ks * kGemmBK, ti.p0, 0, pol_h);
                    ptx::tma_load_2d(sa + 2 * C::A_BYTES, tw, fb, ks * kGemmBK, row_w, pol_w);
                    armed |= 1u << s;
                    parity_bits = (parity_bits & ~(1u << s)) | (ph << s);
                    if (++s == C::STAGES) {
                        s = 0;
                        ph ^= 1u;
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
                const int ksteps = (ti.shared ? a.I_s : a.I) / kGemmBK;
                const int n_f = min(C::NF, a.H - ti.f * C::NF);  // a multiple of 64
                const uint32_t idesc = ptx::idesc_bf16_f32(C::BM, n_f);
                if (!wait_bar(bar_addr(&ctl->tempty[as]), aph ^ 1u, abort_flag, err, code)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + as * C::ACC_COLS;
                for (int ks = 0; ks < ksteps; ++ks) {
                    if (!wait_bar(bar_addr(&ctl->full_a[s]), ph, abort_flag, err, code)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
                    const uint64_t dhi = ptx::smem_desc_sw128(sa);
                    const uint64_t dlo = ptx::smem_desc_sw128(sa + C::A_BYTES);
                    const uint64_t dw = ptx::smem_desc_sw128(sa + 2 * C::A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < kGemmBK / 16; ++kk) {
                        const uint32_t acc = (ks | kk) != 0 ? 1u : 0u;
                        ptx::mma_bf16_ss(d, dhi + 2 * kk, dw + 2 * kk, idesc, acc);
                        ptx::mma_bf16_ss(d, dlo + 2 * kk, dw + 2 * kk, idesc, 1u);
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
    } else if (warp >= 4) {  // ------------------------------ epilogue (warps 4-11)
        // Tokens on TMEM lanes: warp we owns the token rows 32*(warp % 4).. and
        // the features [128*(we / 4), +128) of the tile, drained 32 at a time.
        // Each thread turns 32 consecutive features of its token's y row into
        // y16 codes (64 bytes; its own block exponent) in the warp's staging
        // box, which goes out as one 64-byte x 32-row TMA store; a warp whose
        // token rows are only partly valid stores its valid rows directly. The
        // thread's four exponent bytes go out as one 4-byte store per tile.
        const int we = warp - 4, q = warp & 3, half = we >> 2;
        uint8_t* stg = smem + C::EPI_OFF + we * C::STG_BYTES;
        const uint32_t stg_u32 = ptx::smem_u32(stg);
        const int es = y16_exp_stride(a.H);
        const uint64_t pol_keep = ptx::policy_evict_last();
        int as = 0;
        uint32_t aph = 0;
        const int shared_row0 = a.P;
        int qs = 0;
        uint32_t qph = 0;
        Tile ti;
        while (tq_read(ctl, qs, qph, ti, false, abort_flag, err, code)) {
            if (!wait_bar(bar_addr(&ctl->tfull[as]), aph, abort_flag, err, code)) break;
            ptx::tc_fence_after();
            const int r0 = q * 32;
            const int rows_valid = ti.n_rows - r0;  // token rows of this warp that are real
            const int c_begin = half * (C::NF / 2);
            const int n_f = min(C::NF, a.H - ti.f * C::NF);
            if (rows_valid > 0 && c_begin < n_f) {
                const int row0 = (ti.shared ? shared_row0 + ti.m0 : ti.p0) + r0;
                float scale = 1.f;
                if (ti.shared && lane < rows_valid)
                    scale = 1.f / (1.f + expf(-a.gate_logit[ti.m0 + r0 + lane]));
                const uint32_t tb =
                    tmem_base + (static_cast<uint32_t>(r0) << 16) + as * C::ACC_COLS;
                uint32_t eb = 0;  // the thread's block exponents, one byte per chunk
                for (int col = c_begin; col < c_begin + C::NF / 2; col += 32) {
                    if (col >= n_f) break;
                    const int f0 = ti.f * C::NF + col;
                    uint32_t v[32];
                    ptx::tmem_ld_32x32b_x32(tb + col, v);
                    ptx::tmem_ld_wait();
                    uint32_t mx = 0;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        v[i] = __float_as_uint(__uint_as_float(v[i]) * scale);
                        mx = max(mx, v[i] & 0x7FFFFFFFu);
                    }
                    const uint32_t b = y16_block_exp(mx);
                    eb |= b << (((col - c_begin) / 32) * 8);
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = y16_encode(v[2 * i], b) | (y16_encode(v[2 * i + 1], b) << 16);
                    if (rows_valid >= 32) {
                        if (lane == 0) ptx::bulk_wait_read<0>();  // staging box free again
                        __syncwarp();
                        const uint32_t row_addr = stg_u32 + lane * 64;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            ptx::st_shared_v4u(row_addr + 16 * j, w[4 * j], w[4 * j + 1], w[4 * j + 2],
                                               w[4 * j + 3]);
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (row0 >= a.y_keep_row && row0 < a.P)
                                ptx::tma_store_2d_hint(&maps.st[1], stg_u32, 2 * f0, row0, pol_keep);
                            else
                                ptx::tma_store_2d(&maps.st[1], stg_u32, 2 * f0, row0);
                            ptx::bulk_commit();
                        }
                    } else if (lane < rows_valid) {
                        uint4* dst = reinterpret_cast<uint4*>(
                            reinterpret_cast<uint8_t*>(a.y) + static_cast<size_t>(row0 + lane) * 2 * a.H +
                            2 * f0);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                    }
                }
                // bytes past the row's last block fall into the padding of the stride
                if (lane < rows_valid)
                    *reinterpret_cast<uint32_t*>(a.yexp + static_cast<size_t>(row0 + lane) * es +
                                                 (ti.f * C::NF + c_begin) / kY16Block) = eb;
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_addr(&ctl->tempty[as]));
            if (++as == C::ACC_STAGES) {
                as = 0;
                aph ^= 1u;
            }
        }
        if (lane == 0) ptx::bulk_wait_all();
    }
    gemm_teardown<C>(tmem_base, warp);
}

// =========================================== down, stacked h_hi / h_lo rows
// Tiles of up to 64 tokens of one expert against 256 output features (groups
// too small for 128-token tiles): the MMA's M side stacks the tile's 64 h_hi
// rows over its 64 h_lo rows (one TMA box of the h_hi / h_lo pair) and the
// 256 weight rows are the N side, so one MMA of M = 128, N = 256 covers both
// halves for 256 x 16 weights: half the MMA instructions per weight of the
// weights-on-M form (one MMA of N = BN + rows per 128 x 16 weights), whose
// pace at these widths the MMA instruction rate sets. TMEM lanes 0-63 hold
// W h_hi of the tokens and lanes 64-127 W h_lo: the epilogue warp of lanes
// 64 + 32j.. hands its 32 x 32 values per chunk to the warp of lanes 32j..
// through shared memory (mbarrier hand-offs with bounded waits), which adds
// the two halves in fp32, as the weights-on-M epilogue does, and writes y.
struct DownStk {
    static constexpr int BN = 64;                            // tokens per tile (each half)
    static constexpr int NF = 256;                           // output features per tile (MMA N)
    static constexpr int A_BYTES = 2 * BN * kGemmBK * 2;     // 16 KB: h_hi rows, then h_lo rows
    static constexpr int W_BYTES = NF * kGemmBK * 2;         // 32 KB: weight tile
    static constexpr int STAGE_BYTES = A_BYTES + W_BYTES;
    static constexpr int XCH_BYTES = 32 * 32 * 4;            // one warp pair's hand-off block
    static constexpr int STG_BYTES = 32 * 32 * 4;            // one storing warp's y box (64 B rows used)
    static constexpr int XBAR_OFF = 4 * XCH_BYTES + 4 * STG_BYTES;  // hand-off mbarriers
    static constexpr int EPI_BYTES = XBAR_OFF + 1024;
    static constexpr int CTL_BYTES = 1024;
    static constexpr int STAGES_FIT = (kSmemLimit - 1024 - EPI_BYTES - CTL_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > kStageCap ? kStageCap : STAGES_FIT;
    static constexpr int EPI_OFF = STAGES * STAGE_BYTES;
    static constexpr int CTL_OFF = EPI_OFF + EPI_BYTES;
    static constexpr int SMEM = 1024 + CTL_OFF + CTL_BYTES;
    static constexpr int ACC_COLS = NF;
    static constexpr int A_STAGES = 0;
    static constexpr int CONVERTER_WARPS = 0;
    static constexpr int ACC_STAGES = 2;
    static constexpr int TMEM_COLS = 512;
    static_assert(STAGES >= 3, "pipeline depth");
    static_assert(SMEM <= kSmemLimit, "shared memory budget");
    static_assert(EPI_OFF % 1024 == 0 && STG_BYTES % 1024 == 0, "swizzled staging alignment");
};

__global__ void __launch_bounds__(kThreads, 1)
down_stk_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs a) {
    using C = DownStk;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    Ctl* ctl = reinterpret_cast<Ctl*>(smem + C::CTL_OFF);
    uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + C::EPI_OFF + C::XBAR_OFF);  // [4] full, [4] empty
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ptx::griddep_launch_dependents();
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&maps.w);
        ptx::prefetch_tmap(&maps.ws);
        ptx::prefetch_tmap(&maps.h);
        ptx::prefetch_tmap(&maps.hs);
        ptx::prefetch_tmap(&maps.st[1]);
    }
    if (threadIdx.x == 0)
        for (int i = 0; i < 8; ++i) ptx::mbar_init(bar_addr(&xbar[i]), 1);  // fenced in gemm_setup
    const uint32_t tmem_base = gemm_setup<C>(ctl, warp, 1 + kEpiWarps);
    ptx::griddep_wait();  // h, tile lists and the gate logits come from earlier kernels

    const int R = a.meta[META_RT_DN];
    const int F = (a.H + C::NF - 1) / C::NF;
    const int shared_tiles = ((a.T + C::BN - 1) / C::BN) * F;
    const int num_tiles = R * F + shared_tiles;
    volatile int* abort_flag = &ctl->abort;
    unsigned* err = a.err;
    const unsigned code = ERR_DOWN_TIMEOUT;

    if (warp == 0) {
        if (lane == 0) {  // ---------------------------------- TMA producer
            const uint64_t pol_w = ptx::policy_evict_normal();
            const uint64_t pol_h = ptx::policy_evict_last();  // h rows are re-read per feature block
            int s = 0;
            uint32_t ph = 0, armed = 0, parity_bits = 0;
            bool ok = true;
            TileSched<C::BN> sch;
            Tile ti = sch.start(num_tiles, shared_tiles, F, F, a);
            int qs = 0;
            uint32_t qph = 0;
            ok = tq_publish(ctl, qs, qph, ti, abort_flag, err, code);
            for (; ok && ti.n_rows >= 0;
                 ok = ok && sch.next(ti, a) && tq_publish(ctl, qs, qph, ti, abort_flag, err, code)) {
                sch.prefetch(a);
                const int ksteps = (ti.shared ? a.I_s : a.I) / kGemmBK;
                const CUtensorMap* tw = ti.shared ? &maps.ws : &maps.w;
                const CUtensorMap* th = ti.shared ? &maps.hs : &maps.h;
                // Rows past this expert's H (a ragged last block) read the next
                // expert's rows or zero fill; their columns are never stored.
                const int row_w = (ti.shared ? 0 : ti.e * a.H) + ti.f * C::NF;
                for (int ks = 0; ks < ksteps; ++ks) {
                    if (!wait_bar(bar_addr(&ctl->empty[s]), ph ^ 1u, abort_flag, err, code)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
                    const uint32_t fb = bar_addr(&ctl->full_a[s]);
                    ptx::mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
                    // the tile's 64 h_hi rows, then its 64 h_lo rows (one request);
                    // then 256 weight rows (one request)
                    ptx::tma_load_3d(sa, th, fb, ks * kGemmBK, ti.p0, 0, pol_h);
                    ptx::tma_load_2d(sa + C::A_BYTES, tw, fb, ks * kGemmBK, row_w, pol_w);
                    armed |= 1u << s;
                    parity_bits = (parity_bits & ~(1u << s)) | (ph << s);
                    if (++s == C::STAGES) {
                        s = 0;
                        ph ^= 1u;
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
                const int ksteps = (ti.shared ? a.I_s : a.I) / kGemmBK;
                const int n_f = min(C::NF, a.H - ti.f * C::NF);  // a multiple of 64
                const uint32_t idesc = ptx::idesc_bf16_f32(128, n_f);
                if (!wait_bar(bar_addr(&ctl->tempty[as]), aph ^ 1u, abort_flag, err, code)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + as * C::ACC_COLS;
                for (int ks = 0; ks < ksteps; ++ks) {
                    if (!wait_bar(bar_addr(&ctl->full_a[s]), ph, abort_flag, err, code)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + s * C::STAGE_BYTES);
                    const uint64_t dh = ptx::smem_desc_sw128(sa);
                    const uint64_t dw = ptx::smem_desc_sw128(sa + C::A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < kGemmBK / 16; ++kk)
                        ptx::mma_bf16_ss(d, dh + 2 * kk, dw + 2 * kk, idesc, (ks | kk) != 0 ? 1u : 0u);
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
    } else if (warp >= 4) {  // ------------------------------ epilogue (warps 4-11)
        // Warp (q, half) reads TMEM lanes 32q.. over the columns [128 half, +128)
        // in 32-column chunks. q = 0, 1 (lanes 0-63: W h_hi of tokens 32q..)
        // store; q = 2, 3 (W h_lo of the same tokens) hand their chunk to the
        // warp of q - 2 through block p (its mbarriers xbar[p] full, xbar[4 + p]
        // empty). The storing warp adds the halves, scales shared-expert rows by
        // the gate, and writes y: y16 codes (its own staging box, one TMA store
        // per chunk of 32 full rows, the four exponent bytes of the tile as one
        // 4-byte store) or fp32 rows.
        const int we = warp - 4, q = warp & 3, half = we >> 2;
        const bool store = q < 2;
        const int p = (q & 1) + 2 * half;
        float* xb = reinterpret_cast<float*>(smem + C::EPI_OFF + p * C::XCH_BYTES);
        uint8_t* stg = smem + C::EPI_OFF + 4 * C::XCH_BYTES + p * C::STG_BYTES;
        const uint32_t stg_u32 = ptx::smem_u32(stg);
        const uint32_t xfull = bar_addr(&xbar[p]), xempty = bar_addr(&xbar[4 + p]);
        const int es = y16_exp_stride(a.H);
        uint32_t xph = 0;
        int as = 0;
        uint32_t aph = 0;
        const int shared_row0 = a.P;
        int qs = 0;
        uint32_t qph = 0;
        bool ok = true;
        Tile ti;
        while (ok && tq_read(ctl, qs, qph, ti, false, abort_flag, err, code)) {
            if (!wait_bar(bar_addr(&ctl->tfull[as]), aph, abort_flag, err, code)) break;
            ptx::tc_fence_after();
            const int r0 = (q & 1) * 32;            // this pair's first token row of the tile
            const int rows_valid = ti.n_rows - r0;  // the pair's token rows that are real
            const int c_begin = half * (C::NF / 2);
            const int n_f = min(C::NF, a.H - ti.f * C::NF);
            if (rows_valid > 0 && c_begin < n_f) {
                const int row0 = (ti.shared ? shared_row0 + ti.m0 : ti.p0) + r0;
                float scale = 1.f;
                if (store && ti.shared && lane < rows_valid)
                    scale = 1.f / (1.f + expf(-a.gate_logit[ti.m0 + r0 + lane]));
                const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + as * C::ACC_COLS;
                uint32_t eb = 0;
                for (int col = c_begin; col < c_begin + C::NF / 2; col += 32) {
                    if (col >= n_f) break;
                    uint32_t v[32];
                    ptx::tmem_ld_32x32b_x32(tb + col, v);
                    ptx::tmem_ld_wait();
                    if (!store) {
                        if (!wait_bar(xempty, xph ^ 1u, abort_flag, err, code)) {
                            ok = false;
                            break;
                        }
#pragma unroll
                        for (int c = 0; c < 32; ++c) xb[c * 32 + lane] = __uint_as_float(v[c]);
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(xfull);
                        xph ^= 1u;
                        continue;
                    }
                    if (!wait_bar(xfull, xph, abort_flag, err, code)) {
                        ok = false;
                        break;
                    }
                    float f[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) f[c] = (__uint_as_float(v[c]) + xb[c * 32 + lane]) * scale;
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(xempty);
                    xph ^= 1u;
                    const int f0 = ti.f * C::NF + col;
                    if (a.yexp) {
                        uint32_t mx = 0;
#pragma unroll
                        for (int c = 0; c < 32; ++c) mx = max(mx, __float_as_uint(f[c]) & 0x7FFFFFFFu);
                        const uint32_t b = y16_block_exp(mx);
                        eb |= b << (((col - c_begin) / 32) * 8);
                        uint32_t w[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            w[i] = y16_encode(__float_as_uint(f[2 * i]), b) |
                                   (y16_encode(__float_as_uint(f[2 * i + 1]), b) << 16);
                        if (rows_valid >= 32) {
                            if (lane == 0) ptx::bulk_wait_read<0>();  // staging box free again
                            __syncwarp();
                            const uint32_t row_addr = stg_u32 + lane * 64;
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                ptx::st_shared_v4u(row_addr + 16 * j, w[4 * j], w[4 * j + 1],
                                                   w[4 * j + 2], w[4 * j + 3]);
                            ptx::fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                ptx::tma_store_2d(&maps.st[1], stg_u32, 2 * f0, row0);
                                ptx::bulk_commit();
                            }
                        } else if (lane < rows_valid) {
                            uint4* dst = reinterpret_cast<uint4*>(
                                reinterpret_cast<uint8_t*>(a.y) + static_cast<size_t>(row0 + lane) * 2 * a.H +
                                2 * f0);
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                        }
                    } else if (lane < rows_valid) {
                        float4* dst = reinterpret_cast<float4*>(a.y + static_cast<size_t>(row0 + lane) * a.H + f0);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_float4(f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3]);
                    }
                }
                // bytes past the row's last block fall into the padding of the stride
                if (ok && store && a.yexp && lane < rows_valid)
                    *reinterpret_cast<uint32_t*>(a.yexp + static_cast<size_t>(row0 + lane) * es +
                                                 (ti.f * C::NF + c_begin) / kY16Block) = eb;
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_addr(&ctl->tempty[as]));
            if (++as == C::ACC_STAGES) {
                as = 0;
                aph ^= 1u;
            }
        }
        if (lane == 0) ptx::bulk_wait_all();
    }
    gemm_teardown<C>(tmem_base, warp);
}

cudaError_t launch_down_stk(const GemmMaps& maps, const GemmArgs& a, int max_tiles, int num_sms,
                            cudaStream_t st) {
    using C = DownStk;
    cudaError_t e = cudaFuncSetAttribute(down_stk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM);
    if (e != cudaSuccess) return e;
    const int grid = max_tiles < num_sms ? max_tiles : num_sms;
    if (grid <= 0) return cudaSuccess;
    return launch_kernel(down_stk_kernel, dim3(grid), dim3(kThreads), C::SMEM, st, true, maps, a);
}

template <int BN, bool GU>
cudaError_t launch_bn(const GemmMaps& maps, const GemmArgs& a, int max_tiles, int num_sms,
                      cudaStream_t st) {
    using C = Cfg<BN, GU>;
    void (*kern)(GemmMaps, GemmArgs);
    if constexpr (GU)
        kern = gate_up_kernel<BN>;
    else
        kern = down_kernel<BN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const int grid = max_tiles < num_sms ? max_tiles : num_sms;
    if (grid <= 0) return cudaSuccess;
    return launch_kernel(kern, dim3(grid), dim3(kThreads), C::SMEM, st, true, maps, a);
}

cudaError_t launch_down_ts(const GemmMaps& maps, const GemmArgs& a, int max_tiles, int num_sms,
                           cudaStream_t st) {
    using C = DownTs;
    cudaError_t e = cudaFuncSetAttribute(down_ts_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM);
    if (e != cudaSuccess) return e;
    const int grid = max_tiles < num_sms ? max_tiles : num_sms;
    if (grid <= 0) return cudaSuccess;
    return launch_kernel(down_ts_kernel, dim3(grid), dim3(kThreads), C::SMEM, st, true, maps, a);
}

template <bool GU>
cudaError_t dispatch(int bn, const GemmMaps& maps, const GemmArgs& a, int max_tiles, int num_sms,
                     cudaStream_t st) {
    switch (bn) {
        case 16: return launch_bn<16, GU>(maps, a, max_tiles, num_sms, st);
        case 32: return launch_bn<32, GU>(maps, a, max_tiles, num_sms, st);
        case 64:
            if constexpr (GU) return launch_bn<64, GU>(maps, a, max_tiles, num_sms, st);
            return launch_down_stk(maps, a, max_tiles, num_sms, st);
        case 128:
            if constexpr (GU) return launch_bn<128, GU>(maps, a, max_tiles, num_sms, st);
            return launch_down_ts(maps, a, max_tiles, num_sms, st);
        case 160:
            if constexpr (GU) return launch_bn<160, GU>(maps, a, max_tiles, num_sms, st);
            return cudaErrorInvalidValue;
        case 256:
            if constexpr (GU) return launch_bn<256, GU>(maps, a, max_tiles, num_sms, st);
            return cudaErrorInvalidValue;  // down tiles are at most 128 tokens wide
        default: return cudaErrorInvalidValue;
    }
}

// Self-test of the bounded barrier wait the GEMM roles use: one thread waits
// on an mbarrier that nothing arrives on. The wait must give up after its
// time limit, set `code` in the status word and leave the kernel normally.
__global__ void __launch_bounds__(32, 1) wait_limit_selftest_kernel(unsigned* err) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    ptx::mbar_init(bar_addr(&bar), 1);
    ptx::fence_mbar_init();
    if (wait_bar(bar_addr(&bar), 0u, &abort_flag, err, ERR_GATE_UP_TIMEOUT))
        atomicOr(err, 0x80000000u);  // the wait returned "complete": the test fails
}

}  // namespace

bool gemm_bn_supported(int bn) {
    return bn == 16 || bn == 32 || bn == 64 || bn == 128 || bn == 160 || bn == 256;
}

cudaError_t launch_gate_up(int bn, const GemmMaps& maps, const GemmArgs& a, int max_tiles,
                           int num_sms, cudaStream_t st) {
    return dispatch<true>(bn, maps, a, max_tiles, num_sms, st);
}

cudaError_t launch_wait_limit_selftest(unsigned* err, cudaStream_t st) {
    wait_limit_selftest_kernel<<<1, 32, 0, st>>>(err);
    return cudaGetLastError();
}

cudaError_t launch_down(int bn, const GemmMaps& maps, const GemmArgs& a, int max_tiles,
                        int num_sms, cudaStream_t st) {
    return dispatch<false>(bn, maps, a, max_tiles, num_sms, st);
}

}  // namespace moe
