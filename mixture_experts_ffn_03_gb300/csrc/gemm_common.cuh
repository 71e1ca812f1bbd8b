// Pipeline machinery shared by the grouped expert GEMMs (moe_gemm.cu, bf16
// weights; moe_gemm_mx.cu, MXFP8 weights): tile descriptors and their
// dynamic schedule, the shared-memory control block, bounded mbarrier waits,
// TMEM set-up and the down GEMM's epilogue role.
#pragma once

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per barrier wait
constexpr int kMaxStages = 12;                     // pipeline stage barriers
constexpr int kStageCap = 8;                       // usual pipeline depth cap
constexpr int kSmemLimit = 232448;

constexpr int kEpiWarps = 8;                       // two per TMEM lane quadrant
constexpr int kTileQ = 8;                          // tile descriptors in flight between roles
constexpr int kMaxAStages = 4;                     // TMEM weight stages (MXFP8 GEMMs)
constexpr int kStgBytes = kEpiRows * kEpiCols * 4;  // one staging buffer (2 KB)

struct Tile {
    int shared;  // 1: shared-expert tile
    int e;       // routed expert
    int m0;      // first row inside the group
    int n_rows;  // valid token rows in this tile (1..BN)
    int p0;      // first row in the sorted slot order (routed) or token index (shared)
    int f;       // block of output features (128 rows; gate_up tokens-on-M tiles: NF)
};

struct Ctl {
    uint64_t full_a[kMaxStages];  // TMA bytes landed
    uint64_t full_b[kMaxStages];  // gathered rows landed (gate_up)
    uint64_t empty[kMaxStages];   // MMAs reading the stage completed
    uint64_t tfull[2];            // accumulator ready for the epilogue
    uint64_t tempty[2];           // accumulator drained
    uint64_t drain;               // MMA completion on the abort path
    uint64_t a_full[kMaxAStages]; // converted weight stage written to TMEM (MXFP8 GEMMs)
    uint64_t a_empty[kMaxAStages];// MMAs reading the TMEM weight stage completed
    uint64_t tq_full[kTileQ];     // tile descriptor published
    uint64_t tq_empty[kTileQ];    // tile descriptor read by every consumer role
    Tile tq[kTileQ];              // tile descriptors, in processing order
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Ctl) <= 1024, "control block fits its shared-memory slot");

// Tile order: the shared expert's tiles first (they carry the most tokens
// per tile), then the routed row tiles, the feature blocks of a row tile
// consecutive. A tile index past the end gives the sentinel (n_rows < 0).
__device__ __forceinline__ int4 load_rowtile(int tile, int num_tiles, int shared_tiles, int F,
                                             const GemmArgs& a) {
    if (tile < shared_tiles || tile >= num_tiles) return make_int4(0, 0, 0, 0);
    return a.rowtiles[(tile - shared_tiles) / F];
}

template <int BN>
__device__ __forceinline__ Tile make_tile(int tile, int4 r, int num_tiles, int shared_tiles,
                                          int F, int F_s, const GemmArgs& a) {
    Tile ti;
    if (tile >= num_tiles) {
        ti.shared = 0;
        ti.e = 0;
        ti.m0 = 0;
        ti.n_rows = -1;
        ti.p0 = 0;
        ti.f = 0;
    } else if (tile < shared_tiles) {
        const int rt = tile / F_s;
        ti.f = tile - rt * F_s;
        ti.shared = 1;
        ti.e = 0;
        ti.m0 = rt * BN;
        ti.n_rows = min(BN, a.T - ti.m0);
        ti.p0 = ti.m0;
    } else {
        const int t2 = tile - shared_tiles;
        const int rt = t2 / F;
        ti.f = t2 - rt * F;
        ti.shared = 0;
        ti.e = r.x;
        ti.m0 = r.y;
        ti.n_rows = r.z;
        ti.p0 = r.w;
    }
    return ti;
}

// Dynamic tile scheduling, run by the TMA producer thread: a CTA's first tile
// is blockIdx.x, every further tile is claimed from a global counter. The
// claim and the row-tile load for the next tile are issued one tile ahead, so
// their latency hides behind the current tile's loads.
template <int BN>
struct TileSched {
    int nxt;    // tile after the current one
    int after;  // claim for the tile after nxt (read one tile later)
    int4 raw;   // row-tile entry of nxt
    int num_tiles, shared_tiles, F, F_s;

    __device__ __forceinline__ Tile start(int n_tiles, int s_tiles, int f, int f_s,
                                          const GemmArgs& a) {
        num_tiles = n_tiles;
        shared_tiles = s_tiles;
        F = f;
        F_s = f_s;
        const int first = blockIdx.x;
        nxt = first < num_tiles ? static_cast<int>(gridDim.x) + atomicAdd(a.sched, 1) : num_tiles;
        return make_tile<BN>(first, load_rowtile(first, num_tiles, shared_tiles, F, a), num_tiles,
                             shared_tiles, F, F_s, a);
    }
    // At the start of a tile: claim the tile after next and load next's row tile.
    __device__ __forceinline__ void prefetch(const GemmArgs& a) {
        raw = load_rowtile(nxt, num_tiles, shared_tiles, F, a);
        after = nxt < num_tiles ? static_cast<int>(gridDim.x) + atomicAdd(a.sched, 1) : num_tiles;
    }
    // At the end of a tile: the next tile's descriptor.
    __device__ __forceinline__ bool next(Tile& ti, const GemmArgs& a) {
        ti = make_tile<BN>(nxt, raw, num_tiles, shared_tiles, F, F_s, a);
        nxt = after;
        return true;
    }
};

__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       unsigned* err, unsigned code) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 63u) {
            if (*abort_flag) return false;
            if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicOr(err, code);
                return false;
            }
        }
    }
}

// Wait for phase `parity` of `bar`; false if the CTA is aborting or the wait
// timed out (which starts the abort).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned* err, unsigned code) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, abort_flag, err, code);
}

// Abort-path wait that ignores the abort flag, bounded by the time limit.
__device__ __noinline__ void wait_bounded(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) return;
    }
}

__device__ __forceinline__ uint32_t bar_addr(const uint64_t* b) { return ptx::smem_u32(b); }

// Publish the next tile descriptor (the producer); false on abort or timeout.
__device__ __forceinline__ bool tq_publish(Ctl* ctl, int& s, uint32_t& ph, const Tile& ti,
                                           volatile int* abort_flag, unsigned* err, unsigned code) {
    if (!wait_bar(bar_addr(&ctl->tq_empty[s]), ph ^ 1u, abort_flag, err, code)) return false;
    ctl->tq[s] = ti;
    ptx::mbar_arrive(bar_addr(&ctl->tq_full[s]));  // release: the descriptor is visible
    if (++s == kTileQ) {
        s = 0;
        ph ^= 1u;
    }
    return true;
}

// Read the next tile descriptor (a consumer role; `single` when the role is
// one thread, else the whole warp calls it and lane 0 releases the slot).
// False at the end of the sequence, on abort or on timeout.
__device__ __forceinline__ bool tq_read(Ctl* ctl, int& s, uint32_t& ph, Tile& ti, bool single,
                                        volatile int* abort_flag, unsigned* err, unsigned code) {
    if (!wait_bar(bar_addr(&ctl->tq_full[s]), ph, abort_flag, err, code)) return false;
    ti = ctl->tq[s];
    if (!single) __syncwarp();
    if (single || (threadIdx.x & 31) == 0) ptx::mbar_arrive(bar_addr(&ctl->tq_empty[s]));
    if (++s == kTileQ) {
        s = 0;
        ph ^= 1u;
    }
    return ti.n_rows >= 0;
}

// Common set-up: barriers, TMEM allocation. Returns the TMEM base address.
// C is the kernel's shared-memory / TMEM configuration.
// tq_consumers: warps (or single threads) that read each tile descriptor.
template <class C>
__device__ __forceinline__ uint32_t gemm_setup(Ctl* ctl, int warp, int tq_consumers) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            ptx::mbar_init(bar_addr(&ctl->full_a[s]), 1);
            ptx::mbar_init(bar_addr(&ctl->full_b[s]), 64);
            ptx::mbar_init(bar_addr(&ctl->empty[s]), 1);
        }
        for (int s = 0; s < C::ACC_STAGES; ++s) {
            ptx::mbar_init(bar_addr(&ctl->tfull[s]), 1);
            ptx::mbar_init(bar_addr(&ctl->tempty[s]), kEpiWarps);
        }
        for (int s = 0; s < C::A_STAGES; ++s) {
            ptx::mbar_init(bar_addr(&ctl->a_full[s]), C::CONVERTER_WARPS);
            ptx::mbar_init(bar_addr(&ctl->a_empty[s]), 1);
        }
        ptx::mbar_init(bar_addr(&ctl->drain), 1);
        for (int q = 0; q < kTileQ; ++q) {
            ptx::mbar_init(bar_addr(&ctl->tq_full[q]), 1);
            ptx::mbar_init(bar_addr(&ctl->tq_empty[q]), tq_consumers);
        }
        ctl->abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&ctl->tmem_base), C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    return ctl->tmem_base;
}

template <class C>
__device__ __forceinline__ void gemm_teardown(uint32_t tmem_base, int warp) {
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// Abort path of the TMA producer: wait (bounded) until the last load armed on
// every stage has landed, so no copy is in flight when the CTA exits.
template <int STAGES>
__device__ __forceinline__ void drain_tma(Ctl* ctl, uint32_t armed, uint32_t parity_bits) {
    for (int s = 0; s < STAGES; ++s)
        if (armed & (1u << s)) wait_bounded(bar_addr(&ctl->full_a[s]), (parity_bits >> s) & 1u);
}

// Scale of the tile's weight matrix: the fp32 matrix scale of NVFP4 weights
// (per routed expert, or the shared expert's), 1 for bf16 and MXFP8 weights.
// Bit 0 of Tile::shared marks the shared expert (other bits may tag the tile).
__device__ __forceinline__ float matrix_scale(const GemmArgs& a, const Tile& ti) {
    if (!a.msc) return 1.f;
    return (ti.shared & 1) ? a.msc_s[0] : a.msc[ti.e];
}

// One gate_up tile with the tokens on TMEM lanes (tokens on the MMA's M side,
// NF gate then NF up accumulator columns from `slot`), drained by epilogue
// warp (q, half): it owns the 32 token rows 32q.. and the features
// [NF/2 half, +NF/2) of the tile, and writes h = silu(gate) * up as bf16 hi/lo
// pairs (h_hi = bf16(h), h_lo = bf16(h - h_hi)) with 16-byte stores of its
// own row. Warp-uniform; the whole warp calls it.
template <int NF = kGemmBM>
__device__ __forceinline__ void gate_up_ts_epilogue_tile(const Tile& ti, uint32_t slot, int q,
                                                         int half, int lane, const GemmArgs& a) {
    const int r0 = q * 32;  // first token row of this warp's lane quadrant
    if (r0 >= ti.n_rows) return;
    const bool sh = (ti.shared & 1) != 0;
    const int n_feat = sh ? a.I_s : a.I;
    const bool row_ok = r0 + lane < ti.n_rows;
    const size_t prow = static_cast<size_t>(ti.p0 + r0 + lane) * n_feat;
    __nv_bfloat16* dhi = sh ? a.hs_hi : a.h_hi;
    __nv_bfloat16* dlo = sh ? a.hs_lo : a.h_lo;
    const uint32_t tb = slot + (static_cast<uint32_t>(r0) << 16);
    for (int c = half * (NF / 2); c < (half + 1) * (NF / 2); c += 32) {
        const int fb = ti.f * NF + c;
        if (fb >= n_feat) break;  // I, I_s are multiples of 64
        uint32_t g[32], u[32];
        ptx::tmem_ld_32x32b_x32(tb + c, g);
        ptx::tmem_ld_32x32b_x32(tb + NF + c, u);
        ptx::tmem_ld_wait();
        if (row_ok) {
            uint32_t hi2[16], lo2[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float g0 = __uint_as_float(g[2 * j]);
                const float g1 = __uint_as_float(g[2 * j + 1]);
                const float h0 = __fdividef(g0, 1.f + __expf(-g0)) * __uint_as_float(u[2 * j]);
                const float h1 = __fdividef(g1, 1.f + __expf(-g1)) * __uint_as_float(u[2 * j + 1]);
                const __nv_bfloat162 hp = __floats2bfloat162_rn(h0, h1);
                const __nv_bfloat162 lp =
                    __floats2bfloat162_rn(h0 - __low2float(hp), h1 - __high2float(hp));
                hi2[j] = *reinterpret_cast<const uint32_t*>(&hp);
                lo2[j] = *reinterpret_cast<const uint32_t*>(&lp);
            }
            uint4* phi = reinterpret_cast<uint4*>(dhi + prow + fb);
            uint4* plo = reinterpret_cast<uint4*>(dlo + prow + fb);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                phi[v] = make_uint4(hi2[4 * v], hi2[4 * v + 1], hi2[4 * v + 2], hi2[4 * v + 3]);
                plo[v] = make_uint4(lo2[4 * v], lo2[4 * v + 1], lo2[4 * v + 2], lo2[4 * v + 3]);
            }
        }
    }
}

// One down tile with the weights on M (W h_hi in accumulator columns [0, BN)
// and W h_lo in [BN, 2 BN) from `slot`), drained by epilogue warp (q, half):
// it owns 32 output features (TMEM lanes 32q..) and every other 16-column
// chunk. Shared-expert rows are scaled by their token's gate sigmoid(x .
// w_g), NVFP4 tiles by the matrix scale. y is written as y16 codes when
// a.yexp is set (the warp's 32 features of a row are one block: a warp-wide
// maximum gives its exponent byte), else as fp32. Full chunks go out as TMA
// box stores through st_y[2] (y16 codes, 64 bytes x 16 rows) or st_y[0]
// (fp32), staged in the warp's BUFS buffers at stg (nbuf counts the buffers
// used); ragged tails as plain stores. Warp-uniform.
template <int BN, int BUFS>
__device__ __forceinline__ void down_epilogue_tile(const Tile& ti, uint32_t slot, int q, int half,
                                                   int lane, uint8_t* stg, uint32_t& nbuf,
                                                   const CUtensorMap* st_y, const GemmArgs& a) {
    const bool sh = (ti.shared & 1) != 0;
    const int h0 = ti.f * kGemmBM + q * kEpiCols;  // output feature of lane 0
    const bool warp_valid = h0 < a.H;               // H is a multiple of 64
    const int row0 = sh ? a.P + ti.m0 : ti.p0;
    const float msc = matrix_scale(a, ti);
    const uint32_t tb = slot + (static_cast<uint32_t>(q * 32) << 16);
    for (int c0 = half * kEpiRows; c0 < ti.n_rows; c0 += 2 * kEpiRows) {
        uint32_t v[kEpiRows], vl[kEpiRows];
        ptx::tmem_ld_32x32b_x16(tb + c0, v);        // W h_hi
        ptx::tmem_ld_32x32b_x16(tb + BN + c0, vl);  // W h_lo
        ptx::tmem_ld_wait();
        if (!warp_valid) continue;
        const int rows = min(kEpiRows, ti.n_rows - c0);
        float val[kEpiRows];
#pragma unroll
        for (int n = 0; n < kEpiRows; ++n) {
            val[n] = msc * (__uint_as_float(v[n]) + __uint_as_float(vl[n]));
            if (sh && n < rows) val[n] *= 1.f / (1.f + expf(-a.gate_logit[ti.m0 + c0 + n]));
        }
        if (a.yexp) {
            uint32_t code[kEpiRows], b_row = 0;  // lane n keeps row n's exponent byte
#pragma unroll
            for (int n = 0; n < kEpiRows; ++n) {
                const uint32_t x = __float_as_uint(val[n]);
                const uint32_t b = y16_block_exp(__reduce_max_sync(0xFFFFFFFFu, x & 0x7FFFFFFFu));
                code[n] = y16_encode(x, b);
                if (lane == n) b_row = b;
            }
            if (rows == kEpiRows) {
                const uint32_t bb = nbuf++ % BUFS;
                uint16_t* sc = reinterpret_cast<uint16_t*>(stg + bb * kStgBytes);
                if (lane == 0) ptx::bulk_wait_read<BUFS - 1>();  // buffer bb is free
                __syncwarp();
#pragma unroll
                for (int n = 0; n < kEpiRows; ++n) sc[n * kEpiCols + lane] = static_cast<uint16_t>(code[n]);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::tma_store_2d(st_y + 2, ptx::smem_u32(sc), 2 * h0, row0 + c0);
                    ptx::bulk_commit();
                }
            } else {
                uint16_t* yc = reinterpret_cast<uint16_t*>(a.y);
#pragma unroll
                for (int n = 0; n < kEpiRows; ++n)
                    if (n < rows)
                        yc[static_cast<size_t>(row0 + c0 + n) * a.H + h0 + lane] = static_cast<uint16_t>(code[n]);
            }
            if (lane < rows)
                a.yexp[static_cast<size_t>(row0 + c0 + lane) * y16_exp_stride(a.H) + h0 / kY16Block] =
                    static_cast<uint8_t>(b_row);
        } else if (rows == kEpiRows) {
            const uint32_t b = nbuf++ % BUFS;
            float* sy = reinterpret_cast<float*>(stg + b * kStgBytes);
            if (lane == 0) ptx::bulk_wait_read<BUFS - 1>();  // buffer b is free
            __syncwarp();
#pragma unroll
            for (int n = 0; n < kEpiRows; ++n) sy[n * kEpiCols + lane] = val[n];
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                ptx::tma_store_2d(st_y, ptx::smem_u32(sy), h0, row0 + c0);
                ptx::bulk_commit();
            }
        } else {
#pragma unroll
            for (int n = 0; n < kEpiRows; ++n)
                if (n < rows) a.y[static_cast<size_t>(row0 + c0 + n) * a.H + h0 + lane] = val[n];
        }
    }
}

// Epilogue role of the down GEMMs with the weights on M (warps 4-11): the
// tiles in queue order, each by down_epilogue_tile.
template <class C, int BN>
__device__ __forceinline__ void down_epilogue(uint8_t* smem, Ctl* ctl, uint32_t tmem_base, int warp,
                                              int lane, const CUtensorMap* st_y,
                                              const GemmArgs& a, volatile int* abort_flag,
                                              unsigned* err, unsigned code) {
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
        down_epilogue_tile<BN, C::EPI_BUFS>(ti, tmem_base + as * C::ACC_COLS, q, half, lane, stg,
                                            nbuf, st_y, a);
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

}  // namespace
}  // namespace moe
