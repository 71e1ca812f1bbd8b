// Grouped expert GEMMs with block-quantised expert weights and bf16
// activations. The pages deploy the experts as block-FP8 banks ("qwen3_5_moe
// is TP=1-only ...", first comment) and as NVFP4 (same page, second comment):
//   MXFP8 (OCP Microscaling formats): E4M3 values, one UE8M0 power-of-two
//     scale per 32 consecutive K values of a weight row;
//   NVFP4: E2M1 values (two per byte), one E4M3 scale per 16 consecutive K
//     values, one fp32 scale per weight matrix (applied to the accumulators
//     in the epilogues).
// Either way every block-scaled weight is an exact bf16 number, so the
// products and the fp32 accumulation are the bf16 path's.
//
// The layer's arithmetic is that of moe_gemm.cu (weights on the MMA's M
// side, tokens on N, h as a bf16 hi/lo pair, y as fp32 or, where fp32 y would
// be large, as y16 codes), with the weights
// arriving as one byte (MXFP8) or half a byte (NVFP4) per value:
//   TMA -> shared memory: codes (128-byte swizzle; 64-byte for the NVFP4
//     gate_up rows of 128 values) and their block scales;
//   converter warps: codes -> bf16 (exact), written into TMEM with
//     tcgen05.st, where the MMA reads its A operand (M = 128 weight rows on
//     the 128 lanes, K packed two values per column);
//   MMA: D += A[tmem] * B[smem]^T with B the tokens' rows (gathered hidden
//     rows for gate_up, h panels for down).
// Converted weights never touch shared memory, whose generic traffic is
// then the one-byte codes alone.
//
// Warp roles (640 threads): warp 0 TMA producer and tile scheduler, warp 1
// TMEM owner and MMA issuer, warps 2-3 gather hidden rows (gate_up), warps
// 4-11 epilogue, warps 12-19 converters (warp w converts for TMEM lane
// quadrant w % 4; gate_up: warps 12-15 the gate rows, 16-19 the up rows;
// down: warps 12-15 the first 128 K values of a stage, 16-19 the second).
// Every wait on a pipeline barrier is bounded as in moe_gemm.cu.
#include "gemm_common.cuh"
#include "mxfp8.cuh"

namespace moe {
namespace {

constexpr int kCvtWarps = 8;                                  // two per TMEM lane quadrant
constexpr int kFirstCvtWarp = 4 + kEpiWarps;                  // warp 12
constexpr int kMxThreads = (kFirstCvtWarp + kCvtWarps) * 32;  // 640

// NV: NVFP4 weights (else MXFP8).
template <int BN, bool GU, bool NV>
struct MxCfg {
    // K values per pipeline stage: gate_up 128 (gate and up rows, 32 KB of
    // codes), down 256 (32 KB of codes); each stage is one TMA request of
    // codes, one of scales and (down) one of h.
    static constexpr int KS = GU ? 128 : 256;
    // Code rows (bytes) per stage: MXFP8 gate and up rows of 128 B (128 K), or
    // two 128-B halves per weight row (down); NVFP4 gate and up rows of 64 B
    // (128 K), or one 128-B row per weight row (down, 256 K).
    static constexpr int CODE_ROW = (NV && GU) ? 64 : 128;
    static constexpr int CODE_BYTES = NV ? 2 * kGemmBM * 64 : 2 * kGemmBM * 128;
    static constexpr int SCALE_BLOCK = NV ? 16 : 32;  // K values per block scale
    // Token operand per stage: gate_up two 64-column sub-tiles of BN hidden
    // rows; down four 64-column panels of BN h_hi then BN h_lo rows.
    static constexpr int TOK_BYTES = GU ? 2 * BN * 128 : 4 * 2 * BN * 128;
    // gate_up [KS/SCALE_BLOCK blocks][2 planes][128 rows]; down [KS/SCALE_BLOCK][128]
    static constexpr int SCALE_BYTES = (GU ? 2 : 1) * (KS / SCALE_BLOCK) * kGemmBM;
    static constexpr int TOK_OFF = CODE_BYTES;
    static constexpr int SC_OFF = CODE_BYTES + TOK_BYTES;
    static constexpr int STAGE_BYTES = CODE_BYTES + TOK_BYTES + SCALE_BYTES;
    static constexpr int CTL_BYTES = 1024;
    static constexpr int STAGES_2BUF =
        (kSmemLimit - 1024 - CTL_BYTES - kEpiWarps * 2 * kStgBytes) / STAGE_BYTES;
    static constexpr int STAGES_1BUF =
        (kSmemLimit - 1024 - CTL_BYTES - kEpiWarps * kStgBytes) / STAGE_BYTES;
    static constexpr int EPI_BUFS = (STAGES_2BUF < 4 && STAGES_1BUF > STAGES_2BUF) ? 1 : 2;
    // gate_up writes h with plain stores (decode tiles are ragged anyway), which
    // leaves its shared memory to one more pipeline stage; down stages y.
    static constexpr int EPI_BYTES = GU ? 0 : kEpiWarps * EPI_BUFS * kStgBytes;
    static constexpr int STAGES_FIT = (kSmemLimit - 1024 - CTL_BYTES - EPI_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > kStageCap ? kStageCap : STAGES_FIT;
    static constexpr int CTL_OFF = STAGES * STAGE_BYTES;
    static constexpr int EPI_OFF = CTL_OFF + CTL_BYTES;
    static constexpr int SMEM = 1024 + EPI_OFF + EPI_BYTES;
    // TMEM: two accumulator sets of 2 * BN columns (gate | up, or W h_hi |
    // W h_lo), then weight stages of 128 columns (128 rows x 256 bf16 K
    // values, or gate and up rows x 128 K values each).
    static constexpr int ACC_COLS = 2 * BN;
    static constexpr int ACC_STAGES = 2;
    static constexpr int A_COLS = 128;
    static constexpr int A_BASE = ((2 * ACC_COLS + 127) / 128) * 128;
    static constexpr int A_STAGES_FIT = (512 - A_BASE) / A_COLS;
    static constexpr int A_STAGES = A_STAGES_FIT > kMaxAStages ? kMaxAStages : A_STAGES_FIT;
    static constexpr int TMEM_COLS = 512;
    static constexpr int CONVERTER_WARPS = kCvtWarps;
    static_assert(STAGES >= 2 && A_STAGES >= 2, "pipeline needs two stages");
    static_assert(SMEM <= kSmemLimit, "shared memory budget");
    static_assert(STAGE_BYTES % 1024 == 0 && TOK_OFF % 1024 == 0 && (BN * 128) % 1024 == 0,
                  "swizzled tiles start on 1024-byte boundaries");
    static_assert(BN == 16 || BN == 32 || BN == 64, "quantised-weight tile widths");
    static_assert(SCALE_BYTES % 1024 == 0, "stage parts stay 1024-byte aligned");
};

// One converter thread's share of a stage: the 128 K values (8 chunks of 16
// codes, 128-byte swizzled row `crow` of the stage's code tile) of one weight
// row, scaled by the scale bytes at shared address sc, sc + sc_stride, ...
// (one per 32 values), written to TMEM columns ta .. ta + 63 of this warp's
// lane quadrant. All eight 16-byte loads and the four scale loads are issued
// before the first conversion.
__device__ __forceinline__ void convert_row(uint32_t codes, int crow, uint32_t sc, int sc_stride,
                                            uint32_t ta) {
    const uint32_t row = codes + static_cast<uint32_t>(crow) * 128u;
    const uint32_t swz = static_cast<uint32_t>(crow & 7);
    uint4 v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) v[c] = ptx::ld_shared_v4u(row + ((c ^ swz) << 4));
    uint32_t s[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) s[j] = ptx::ld_shared_u8(sc + j * sc_stride);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t out[16];
        uint32_t lo[8], hi[8];
        mx_dequant16(v[2 * j], s[j], lo);
        mx_dequant16(v[2 * j + 1], s[j], hi);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            out[i] = lo[i];
            out[8 + i] = hi[i];
        }
        ptx::tmem_st_32x32b_x16(ta + 16 * j, out);
    }
}

// NVFP4: one converter thread's share of a stage, the 128 K values (4 chunks
// of 32 codes starting at chunk c_first of the code row at shared address
// `row`, chunk c at position (c ^ swz)) of one weight row, scaled by the 8
// E4M3 scale bytes at sc, sc + sc_stride, ... (one per 16 values), written
// to TMEM columns ta .. ta + 63. All loads are issued before the first
// conversion.
__device__ __forceinline__ void convert_row_nv(uint32_t row, uint32_t swz, int c_first,
                                               uint32_t sc, int sc_stride, uint32_t ta) {
    uint4 v[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
        v[c] = ptx::ld_shared_v4u(row + ((static_cast<uint32_t>(c_first + c) ^ swz) << 4));
    uint32_t s[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j] = ptx::ld_shared_u8(sc + j * sc_stride);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t out[16];
        nv_dequant32(v[c], e4m3_to_bf16x2(s[2 * c]), e4m3_to_bf16x2(s[2 * c + 1]), out);
        ptx::tmem_st_32x32b_x16(ta + 16 * c, out);
    }
}

// Converter role, shared by both GEMMs. Per stage: wait for the codes and a
// free TMEM weight stage, convert, make the TMEM writes visible to the MMA
// issuer and release the stage to it.
template <class C, bool GU, bool NV>
__device__ __forceinline__ void converter_role(uint8_t* smem, Ctl* ctl, uint32_t tmem_base,
                                               int warp, int lane, const GemmArgs& a,
                                               volatile int* abort_flag, unsigned* err,
                                               unsigned code) {
    const int cw = warp - kFirstCvtWarp, q = warp & 3, part = cw >> 2;
    const int r = q * 32 + lane;  // weight row of the tile = TMEM lane
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    int s = 0, t = 0;
    uint32_t ph = 0, tph = 0;
    int qs = 0;
    uint32_t qph = 0;
    Tile ti;
    bool ok = true;
    while (ok && tq_read(ctl, qs, qph, ti, false, abort_flag, err, code)) {
        const int K = GU ? a.H : (ti.shared ? a.I_s : a.I);
        const int ksteps = (K + C::KS - 1) / C::KS;
        for (int ks = 0; ks < ksteps; ++ks) {
            if (!wait_bar(bar_addr(&ctl->full_a[s]), ph, abort_flag, err, code) ||
                !wait_bar(bar_addr(&ctl->a_empty[t]), tph ^ 1u, abort_flag, err, code)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            uint8_t* st = smem + s * C::STAGE_BYTES;
            const uint32_t codes = ptx::smem_u32(st);
            const uint32_t ta = lane_base + C::A_BASE + t * C::A_COLS + part * 64;
            if constexpr (NV && GU) {
                // 64-byte rows [0, 128) gate, [128, 256) up (64-byte swizzle: chunk c of
                // row p at c ^ ((p >> 1) & 3)); scales [block][plane][row]
                const int p = part * kGemmBM + r;
                convert_row_nv(codes + static_cast<uint32_t>(p) * 64u,
                               static_cast<uint32_t>((p >> 1) & 3), 0,
                               codes + C::SC_OFF + part * 128 + r, 256, ta);
            } else if constexpr (NV) {
                // 128-byte row r holds the stage's 256 K values; this part's chunks are
                // 4 part .. 4 part + 3; scales [block][row]
                convert_row_nv(codes + static_cast<uint32_t>(r) * 128u, static_cast<uint32_t>(r & 7),
                               4 * part, codes + C::SC_OFF + (part * 8) * 128 + r, 128, ta);
            } else if constexpr (GU) {
                // rows [0, 128) gate, [128, 256) up; scales [block][plane][row]
                convert_row(codes, part * kGemmBM + r, codes + C::SC_OFF + part * 128 + r, 256, ta);
            } else {
                // code row 2r + part = K values [128 part, 128 part + 128) of row r;
                // scales [block][row]
                convert_row(codes, 2 * r + part, codes + C::SC_OFF + (part * 4) * 128 + r, 128, ta);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_addr(&ctl->a_full[t]));
            if (++s == C::STAGES) {
                s = 0;
                ph ^= 1u;
            }
            if (++t == C::A_STAGES) {
                t = 0;
                tph ^= 1u;
            }
        }
    }
}

// ================================================================ gate_up
template <int BN, bool NV>
__global__ void __launch_bounds__(kMxThreads, 1)
gate_up_mx_kernel(const __grid_constant__ MxMaps maps, const GemmArgs a) {
    using C = MxCfg<BN, true, NV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    Ctl* ctl = reinterpret_cast<Ctl*>(smem + C::CTL_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ptx::griddep_launch_dependents();
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&maps.w);
        ptx::prefetch_tmap(&maps.ws);
        ptx::prefetch_tmap(&maps.sc);
        ptx::prefetch_tmap(&maps.scs);
    }
    const uint32_t tmem_base = gemm_setup<C>(ctl, warp, 1 + 2 + kEpiWarps + kCvtWarps);
    ptx::griddep_wait();  // routing, tile lists and the slot order come from earlier kernels

    const int R = a.meta[META_RT_GU];
    const int F = a.I / kGemmBM, F_s = a.I_s / kGemmBM;
    const int shared_tiles = ((a.T + BN - 1) / BN) * F_s;
    const int num_tiles = R * F + shared_tiles;
    const int ksteps = a.H / C::KS;
    volatile int* abort_flag = &ctl->abort;
    unsigned* err = a.err;
    const unsigned code = ERR_GATE_UP_TIMEOUT;

    if (warp == 0) {
        if (lane == 0) {  // ---------------------------------- TMA producer
            const uint64_t pol = ptx::policy_evict_normal();
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
                const CUtensorMap* tw = ti.shared ? &maps.ws : &maps.w;
                const CUtensorMap* tsc = ti.shared ? &maps.scs : &maps.sc;
                const int row_g = (ti.shared ? 0 : ti.e * 2 * a.I) + ti.f * kGemmBM;
                const int blk0 = ti.shared ? 0 : ti.e * (a.H / C::SCALE_BLOCK);
                for (int ks = 0; ks < ksteps; ++ks) {
                    if (!wait_bar(bar_addr(&ctl->empty[s]), ph ^ 1u, abort_flag, err, code)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + s * C::STAGE_BYTES;
                    const uint32_t fb = bar_addr(&ctl->full_a[s]);
                    ptx::mbar_arrive_expect_tx(fb, C::CODE_BYTES + C::SCALE_BYTES);
                    // x in bytes: 128 K values are 128 (MXFP8) or 64 (NVFP4) bytes
                    ptx::tma_load_3d(ptx::smem_u32(st), tw, fb, ks * C::CODE_ROW, row_g, 0, pol);
                    ptx::tma_load_3d(ptx::smem_u32(st + C::SC_OFF), tsc, fb, ti.f * kGemmBM, 0,
                                     blk0 + ks * (C::KS / C::SCALE_BLOCK), pol);
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
            int s = 0, as = 0, t = 0;
            uint32_t ph = 0, aph = 0, tph = 0;
            bool ok = true;
            int qs = 0;
            uint32_t qph = 0;
            Tile ti;
            while (ok && tq_read(ctl, qs, qph, ti, true, abort_flag, err, code)) {
                const int n_mma = max(16, (ti.n_rows + 15) & ~15);
                const uint32_t idesc = ptx::idesc_bf16_f32(kGemmBM, n_mma);
                if (!wait_bar(bar_addr(&ctl->tempty[as]), aph ^ 1u, abort_flag, err, code)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_gate = tmem_base + as * C::ACC_COLS;
                const uint32_t d_up = d_gate + BN;
                for (int ks = 0; ks < ksteps; ++ks) {
                    if (!wait_bar(bar_addr(&ctl->a_full[t]), tph, abort_flag, err, code) ||
                        !wait_bar(bar_addr(&ctl->full_a[s]), ph, abort_flag, err, code) ||
                        !wait_bar(bar_addr(&ctl->full_b[s]), ph, abort_flag, err, code)) {
                        ok = false;
                        break;
                    }
                    ptx::fence_proxy_async_smem();  // gathered rows were written by cp.async
                    ptx::tc_fence_after();
                    const uint32_t a_gate = tmem_base + C::A_BASE + t * C::A_COLS;
                    const uint32_t sb = ptx::smem_u32(smem + s * C::STAGE_BYTES + C::TOK_OFF);
#pragma unroll
                    for (int kk = 0; kk < C::KS / 16; ++kk) {
                        const uint32_t acc = (ks | kk) != 0 ? 1u : 0u;
                        // 64-column sub-tile kk / 4 of the token rows, +32 bytes per K slice
                        const uint64_t db = ptx::smem_desc_sw128(sb + (kk >> 2) * (BN * 128)) +
                                            2 * (kk & 3);
                        ptx::mma_bf16_ts(d_gate, a_gate + 8 * kk, db, idesc, acc);
                        ptx::mma_bf16_ts(d_up, a_gate + 64 + 8 * kk, db, idesc, acc);
                    }
                    ptx::mma_commit(bar_addr(&ctl->empty[s]));
                    ptx::mma_commit(bar_addr(&ctl->a_empty[t]));
                    if (++s == C::STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (++t == C::A_STAGES) {
                        t = 0;
                        tph ^= 1u;
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
        // As in moe_gemm.cu, for the two 64-column sub-tiles of a stage.
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
            uint32_t trow[RPT];
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                const int r = r_first + 8 * j;
                uint32_t tok = 0;
                if (r < ti.n_rows) tok = ti.shared ? ti.m0 + r : a.perm[ti.p0 + r] / a.k;
                trow[j] = tok;
            }
            const __nv_bfloat16* col = a.hidden + c * 8;
            for (int ks = 0; ks < ksteps; ++ks) {
                if (!wait_bar(bar_addr(&ctl->empty[s]), ph ^ 1u, abort_flag, err, code)) {
                    ok = false;
                    break;
                }
                const uint32_t sb = ptx::smem_u32(smem + s * C::STAGE_BYTES + C::TOK_OFF);
#pragma unroll
                for (int sub = 0; sub < 2; ++sub) {
                    const __nv_bfloat16* src = col + ks * C::KS + sub * 64;
#pragma unroll
                    for (int j = 0; j < RPT; ++j) {
                        const int r = r_first + 8 * j;
                        if (r < ti.n_rows)
                            ptx::cp_async_16(sb + sub * (BN * 128) + r * 128 + swz,
                                             src + static_cast<size_t>(trow[j]) * a.H);
                    }
                }
                ptx::cp_async_arrive_noinc(bar_addr(&ctl->full_b[s]));
                if (++s == C::STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        ptx::cp_async_wait_all();
    } else if (warp < kFirstCvtWarp) {  // -------------------- epilogue (warps 4-11)
        // As the gate_up epilogue with the weights on M in moe_gemm.cu, with h
        // written with plain stores into 64-column panels: warp we drains TMEM
        // lanes 32*(warp % 4) (32 intermediate features, one per lane) for the
        // 16-token chunks 16*(we / 4) + 32*j; a warp's stores of one token row
        // are 64 contiguous bytes.
        const int we = warp - 4, q = warp & 3, half = we >> 2;
        int as = 0;
        uint32_t aph = 0;
        int qs = 0;
        uint32_t qph = 0;
        Tile ti;
        while (tq_read(ctl, qs, qph, ti, false, abort_flag, err, code)) {
            if (!wait_bar(bar_addr(&ctl->tfull[as]), aph, abort_flag, err, code)) break;
            ptx::tc_fence_after();
            const int i = ti.f * kGemmBM + q * kEpiCols + lane;  // this lane's feature (< I or I_s)
            const size_t P = ti.shared ? static_cast<size_t>(a.T)
                                       : static_cast<size_t>(a.T) * a.k;
            __nv_bfloat16* panel = (ti.shared ? a.hs_hi : a.h_hi) +
                                   static_cast<size_t>(i >> 6) * 2 * P * 64 + (i & 63);
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + as * C::ACC_COLS;
            const float msc = matrix_scale(a, ti);  // NVFP4 matrix scale (1 for MXFP8)
            for (int c0 = half * kEpiRows; c0 < ti.n_rows; c0 += 2 * kEpiRows) {
                uint32_t g[kEpiRows], u[kEpiRows];
                ptx::tmem_ld_32x32b_x16(tb + c0, g);
                ptx::tmem_ld_32x32b_x16(tb + BN + c0, u);
                ptx::tmem_ld_wait();
                const int rows = min(kEpiRows, ti.n_rows - c0);
#pragma unroll
                for (int n = 0; n < kEpiRows; ++n) {
                    if (n < rows) {
                        const float gv = msc * __uint_as_float(g[n]);
                        const float h = __fdividef(gv, 1.f + __expf(-gv)) * (msc * __uint_as_float(u[n]));
                        const __nv_bfloat16 hi = __float2bfloat16_rn(h);
                        const size_t o = static_cast<size_t>(ti.p0 + c0 + n) * 64;
                        panel[o] = hi;
                        panel[o + P * 64] = __float2bfloat16_rn(h - __bfloat162float(hi));
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
    } else {  // --------------------------------------------- converters (warps 12-19)
        converter_role<C, true, NV>(smem, ctl, tmem_base, warp, lane, a, abort_flag, err, code);
    }
    gemm_teardown<C>(tmem_base, warp);
}

// =================================================================== down
template <int BN, bool NV>
__global__ void __launch_bounds__(kMxThreads, 1)
down_mx_kernel(const __grid_constant__ MxMaps maps, const GemmArgs a) {
    using C = MxCfg<BN, false, NV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    Ctl* ctl = reinterpret_cast<Ctl*>(smem + C::CTL_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ptx::griddep_launch_dependents();
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&maps.w);
        ptx::prefetch_tmap(&maps.ws);
        ptx::prefetch_tmap(&maps.sc);
        ptx::prefetch_tmap(&maps.scs);
        ptx::prefetch_tmap(&maps.h);
        ptx::prefetch_tmap(&maps.hs);
    }
    const uint32_t tmem_base = gemm_setup<C>(ctl, warp, 1 + kEpiWarps + kCvtWarps);
    ptx::griddep_wait();  // h, tile lists and the gate logits come from earlier kernels

    const int R = a.meta[META_RT_DN];
    const int F = a.H / kGemmBM;
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
                const int K = ti.shared ? a.I_s : a.I;
                const int ksteps = (K + C::KS - 1) / C::KS;
                const CUtensorMap* tw = ti.shared ? &maps.ws : &maps.w;
                const CUtensorMap* tsc = ti.shared ? &maps.scs : &maps.sc;
                const CUtensorMap* th = ti.shared ? &maps.hs : &maps.h;
                const int row_w = (ti.shared ? 0 : ti.e * a.H) + ti.f * kGemmBM;
                const int blk0 = ti.shared ? 0 : ti.e * (a.I / C::SCALE_BLOCK);
                for (int ks = 0; ks < ksteps; ++ks) {
                    if (!wait_bar(bar_addr(&ctl->empty[s]), ph ^ 1u, abort_flag, err, code)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + s * C::STAGE_BYTES;
                    const uint32_t fb = bar_addr(&ctl->full_a[s]);
                    ptx::mbar_arrive_expect_tx(fb, C::CODE_BYTES + C::TOK_BYTES + C::SCALE_BYTES);
                    // 128 rows x 256 K values (K past the end reads as zero codes)
                    if constexpr (NV)
                        ptx::tma_load_2d(ptx::smem_u32(st), tw, fb, ks * 128, row_w, pol_w);
                    else
                        ptx::tma_load_3d(ptx::smem_u32(st), tw, fb, 0, 2 * ks, row_w, pol_w);
                    ptx::tma_load_2d(ptx::smem_u32(st + C::SC_OFF), tsc, fb, ti.f * kGemmBM,
                                     blk0 + ks * (C::KS / C::SCALE_BLOCK), pol_w);
                    // four 64-column panels of the tile's h_hi and h_lo rows
                    ptx::tma_load_4d(ptx::smem_u32(st + C::TOK_OFF), th, fb, 0, ti.p0, 0, 4 * ks,
                                     pol_h);
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
            int s = 0, as = 0, t = 0;
            uint32_t ph = 0, aph = 0, tph = 0;
            bool ok = true;
            int qs = 0;
            uint32_t qph = 0;
            Tile ti;
            while (ok && tq_read(ctl, qs, qph, ti, true, abort_flag, err, code)) {
                const int K = ti.shared ? a.I_s : a.I;
                const int ksteps = (K + C::KS - 1) / C::KS;
                // N = the BN h_hi rows and the tile's h_lo rows of each panel:
                // accumulator columns [0, BN) hold W h_hi, [BN, BN + rows) W h_lo.
                const int n_mma = BN + max(16, (ti.n_rows + 15) & ~15);
                const uint32_t idesc = ptx::idesc_bf16_f32(kGemmBM, n_mma);
                if (!wait_bar(bar_addr(&ctl->tempty[as]), aph ^ 1u, abort_flag, err, code)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + as * C::ACC_COLS;
                for (int ks = 0; ks < ksteps; ++ks) {
                    if (!wait_bar(bar_addr(&ctl->a_full[t]), tph, abort_flag, err, code) ||
                        !wait_bar(bar_addr(&ctl->full_a[s]), ph, abort_flag, err, code)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a_w = tmem_base + C::A_BASE + t * C::A_COLS;
                    const uint32_t sh = ptx::smem_u32(smem + s * C::STAGE_BYTES + C::TOK_OFF);
#pragma unroll
                    for (int kk = 0; kk < C::KS / 16; ++kk) {
                        const uint32_t acc = (ks | kk) != 0 ? 1u : 0u;
                        const uint64_t dh = ptx::smem_desc_sw128(sh + (kk >> 2) * (2 * BN * 128)) +
                                            2 * (kk & 3);
                        ptx::mma_bf16_ts(d, a_w + 8 * kk, dh, idesc, acc);
                    }
                    ptx::mma_commit(bar_addr(&ctl->empty[s]));
                    ptx::mma_commit(bar_addr(&ctl->a_empty[t]));
                    if (++s == C::STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (++t == C::A_STAGES) {
                        t = 0;
                        tph ^= 1u;
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
    } else if (warp < 4) {
        // no row gather: h arrives by TMA
    } else if (warp < kFirstCvtWarp) {  // -------------------- epilogue (warps 4-11)
        down_epilogue<C, BN>(smem, ctl, tmem_base, warp, lane, &maps.st[0], a, abort_flag, err,
                             code);
    } else {  // --------------------------------------------- converters (warps 12-19)
        converter_role<C, false, NV>(smem, ctl, tmem_base, warp, lane, a, abort_flag, err, code);
    }
    gemm_teardown<C>(tmem_base, warp);
}

template <int BN, bool GU, bool NV>
cudaError_t launch_mx_bn(const MxMaps& maps, const GemmArgs& a, int max_tiles, int num_sms,
                         cudaStream_t st) {
    using C = MxCfg<BN, GU, NV>;
    void (*kern)(MxMaps, GemmArgs);
    if constexpr (GU)
        kern = gate_up_mx_kernel<BN, NV>;
    else
        kern = down_mx_kernel<BN, NV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const int grid = max_tiles < num_sms ? max_tiles : num_sms;
    if (grid <= 0) return cudaSuccess;
    return launch_kernel(kern, dim3(grid), dim3(kMxThreads), C::SMEM, st, true, maps, a);
}

template <bool GU, bool NV>
cudaError_t dispatch_mx(int bn, const MxMaps& maps, const GemmArgs& a, int max_tiles, int num_sms,
                        cudaStream_t st) {
    switch (bn) {
        case 16: return launch_mx_bn<16, GU, NV>(maps, a, max_tiles, num_sms, st);
        case 32: return launch_mx_bn<32, GU, NV>(maps, a, max_tiles, num_sms, st);
        case 64: return launch_mx_bn<64, GU, NV>(maps, a, max_tiles, num_sms, st);
        default: return cudaErrorInvalidValue;
    }
}

// One thread per 16 codes of a row: the same conversion the GEMMs' converter
// warps run, written out as bf16.
__global__ void mxfp8_dequant_kernel(const uint8_t* __restrict__ codes,
                                     const uint8_t* __restrict__ scales, int rows, int cols,
                                     __nv_bfloat16* __restrict__ out) {
    const int chunks = cols / 16;
    const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<size_t>(rows) * chunks) return;
    const int r = static_cast<int>(idx / chunks), c = static_cast<int>(idx % chunks);
    const uint4 v = *reinterpret_cast<const uint4*>(codes + static_cast<size_t>(r) * cols + c * 16);
    const uint32_t s = scales[static_cast<size_t>(c / 2) * rows + r];
    uint32_t o[8];
    mx_dequant16(v, s, o);
    uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(r) * cols + c * 16);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// NVFP4: one thread per 32 values (16 code bytes) of a row, the converter
// warps' conversion, written out as bf16 (without the matrix scale).
__global__ void nvfp4_dequant_kernel(const uint8_t* __restrict__ codes,
                                     const uint8_t* __restrict__ scales, int rows, int cols,
                                     __nv_bfloat16* __restrict__ out) {
    const int chunks = cols / 32;
    const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<size_t>(rows) * chunks) return;
    const int r = static_cast<int>(idx / chunks), c = static_cast<int>(idx % chunks);
    const uint4 v =
        *reinterpret_cast<const uint4*>(codes + static_cast<size_t>(r) * (cols / 2) + c * 16);
    const uint32_t s0 = scales[static_cast<size_t>(2 * c) * rows + r];
    const uint32_t s1 = scales[static_cast<size_t>(2 * c + 1) * rows + r];
    uint32_t o[16];
    nv_dequant32(v, e4m3_to_bf16x2(s0), e4m3_to_bf16x2(s1), o);
    uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(r) * cols + c * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
}

}  // namespace

bool gemm_mx_bn_supported(int bn) { return bn == 16 || bn == 32 || bn == 64; }

cudaError_t launch_gate_up_mx(int bn, bool nvfp4, const MxMaps& maps, const GemmArgs& a,
                              int max_tiles, int num_sms, cudaStream_t st) {
    return nvfp4 ? dispatch_mx<true, true>(bn, maps, a, max_tiles, num_sms, st)
                 : dispatch_mx<true, false>(bn, maps, a, max_tiles, num_sms, st);
}

cudaError_t launch_down_mx(int bn, bool nvfp4, const MxMaps& maps, const GemmArgs& a,
                           int max_tiles, int num_sms, cudaStream_t st) {
    return nvfp4 ? dispatch_mx<false, true>(bn, maps, a, max_tiles, num_sms, st)
                 : dispatch_mx<false, false>(bn, maps, a, max_tiles, num_sms, st);
}

cudaError_t launch_mxfp8_dequant(const uint8_t* codes, const uint8_t* scales, int rows, int cols,
                                 __nv_bfloat16* out, cudaStream_t st) {
    const size_t n = static_cast<size_t>(rows) * (cols / 16);
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    const size_t blocks = (n + threads - 1) / threads;
    if (blocks > 0x7FFFFFFFu) return cudaErrorInvalidValue;
    mxfp8_dequant_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(codes, scales, rows,
                                                                            cols, out);
    return cudaGetLastError();
}

cudaError_t launch_nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, int rows, int cols,
                                 __nv_bfloat16* out, cudaStream_t st) {
    const size_t n = static_cast<size_t>(rows) * (cols / 32);
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    const size_t blocks = (n + threads - 1) / threads;
    if (blocks > 0x7FFFFFFFu) return cudaErrorInvalidValue;
    nvfp4_dequant_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(codes, scales, rows,
                                                                            cols, out);
    return cudaGetLastError();
}
}  // namespace moe
