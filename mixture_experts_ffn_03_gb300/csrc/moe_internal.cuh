// Internal interfaces between the host driver (moe_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <utility>

namespace moe {

// Launch `kern` on `st`; with `pdl`, as a programmatic dependent launch so its
// CTAs can be scheduled (and run their set-up) while the previous kernel in
// the stream drains. Kernels launched this way call griddep_wait() before
// reading anything the previous kernel wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Launch `kern` on `st` as a cooperative launch: every CTA of the grid is
// resident at once (the launch fails rather than queueing CTAs behind others),
// which a kernel whose CTAs wait on one another needs.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_cooperative(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Device status word bits (workspace status block, word 0).
enum : unsigned {
    ERR_GATE_UP_TIMEOUT = 1u << 0,
    ERR_DOWN_TIMEOUT = 1u << 1,
    ERR_ROUTER_TIMEOUT = 1u << 2,
    ERR_EP_COUNTS = 1u << 3,      // received-row counts inconsistent (expert parallelism)
};

// Status block layout (int32 words at the start of the workspace).
enum : int {
    META_ERR = 0,          // device error flags
    META_RT_GU = 1,        // routed row tiles of the gate_up GEMM
    META_RT_DN = 2,        // routed row tiles of the down GEMM
    META_TICKET = 3,       // block-completion counter of the routing launch
    META_SCHED_GU = 4,     // tiles claimed by the gate_up GEMM's CTAs (past their first)
    META_SCHED_DN = 5,     // tiles claimed by the down GEMM's CTAs
    META_PERMUTED = 6,     // whole-layer launch: the permute is written
    META_DONE = 7,         // whole-layer launch: CTAs whose expert tiles are all done
    META_WORDS = 64,
};

constexpr int kMaxExperts = 1024;       // routed experts per layer at most
constexpr int kRouteWarps = 8;          // tokens per route block (one warp each)
// 64-K chunks per pipeline stage (one TMA request each for weights and h) of
// the bf16 down GEMM with the weights on M (down_kernel).
constexpr int kDownChunks = 2;
constexpr int kSmallSlots = 2048;       // T*k up to which the routing launch also permutes
constexpr int kCountTokens = 256;       // tokens per histogram block
constexpr int kGemmBM = 128;            // weight rows (output features) per tile
constexpr int kGemmBK = 64;             // K elements per pipeline stage
// Intermediate features per gate_up tile (gate and up rows each) in the
// tokens-on-M kernel for BN-token tiles: decode-sized tiles take 64, so that
// the weight stream is cut into twice as many tiles and the last CTAs to run
// out of work finish closer together; wider tiles take 128.
constexpr int gate_up_ts_features(int bn) { return bn <= 32 ? 64 : 128; }
constexpr int kEpiRows = 16;            // token rows per epilogue store box
constexpr int kEpiCols = 32;            // output columns per epilogue warp (one TMEM lane each)

// y rows of the tokens-on-M down GEMM, read by the combine ("y16"): each
// block of 32 consecutive values of a row has one exponent byte b, the
// biased fp32 exponent of the block's largest magnitude minus 13, clamped to
// [1, 240]. With D = 2^(b - 127), a value v is stored as 16 bits: its sign
// and |v| + D rounded to a 12-bit significand (nearest even), as 4 exponent
// bits counted from b and 11 fraction bits. Decoding adds b back and
// subtracts D, exactly. The error is at most 2^-12 (|v| + D) (a 12-bit
// significand; D is 2^-13 to 2^-14 of the block's largest magnitude, so
// small values get an absolute step of at most 2^-11 D), and zero is
// exact. A block holding an infinity
// or a NaN gets b = 240: those decode as themselves, its finite values
// below 2^114 as zero. Layout: the codes [rows][H] (2H-byte rows), then the
// exponent plane [rows][y16_exp_stride(H)] bytes.
constexpr int kY16Block = 32;
__host__ __device__ constexpr int y16_exp_stride(int H) { return (H / kY16Block + 3) & ~3; }

#ifdef __CUDACC__
// Exponent byte of a block whose largest |value| has the fp32 bits
// `max_abs_bits` (an integer maximum of the values' bits without the sign,
// so infinities and NaNs rank highest).
__device__ __forceinline__ uint32_t y16_block_exp(uint32_t max_abs_bits) {
    const int e = static_cast<int>(max_abs_bits >> 23) - 13;
    return static_cast<uint32_t>(e < 1 ? 1 : (e > 240 ? 240 : e));
}
// 16-bit code of the fp32 value with bits x in a block with exponent byte b.
__device__ __forceinline__ uint32_t y16_encode(uint32_t x, uint32_t b) {
    const uint32_t ax = x & 0x7FFFFFFFu;
    // |v| + D rounded to fp32, then to 12 significant bits (the first
    // rounding moves it by at most 2^-13 of the second one's step)
    const uint32_t c = __float_as_uint(__uint_as_float(ax) + __uint_as_float(b << 23));
    uint32_t em = ((c + 0x7FFu + ((c >> 12) & 1u)) >> 12) - (b << 11);
    if (ax > 0x7F800000u) em = 0x7C00u;  // NaN: all-ones exponent, nonzero fraction
    return em | ((x >> 16) & 0x8000u);
}
__device__ __forceinline__ float y16_decode(uint32_t u, uint32_t b) {
    const float f = __uint_as_float(((u & 0x7FFFu) << 12) + (b << 23)) - __uint_as_float(b << 23);
    return __uint_as_float(__float_as_uint(f) | ((u & 0x8000u) << 16));
}
#endif

// Where the routing kernels read the logits: the sum, in order, of `parts`
// fp32 arrays [T, E] spaced part_stride floats apart (parts = 1: the caller's
// logits; more: the router GEMM's split-K partial sums). `out` (optional)
// receives the summed logits.
struct LogitSrc {
    const float* p;
    int parts;
    size_t part_stride;
    float* out;
};

// Routing, histogram/scan, scatter and combine (moe_route.cu). With `pdl` the
// routing launch is a programmatic dependent of the previous kernel (the
// router GEMM) and waits for it before reading the logits.
bool route_small_fits(int T, int E, int k);
cudaError_t launch_route_permute(int T, int H, int E, int k, int score_fn, int bn_gu, int bn_dn,
                                 const LogitSrc& logits, bool pdl, const __nv_bfloat16* hidden,
                                 const __nv_bfloat16* w_g, int* topk_ids, float* topk_w,
                                 float* gate_logit, int* counts, int* offsets, int* perm,
                                 int* inv, int4* rt_gu, int4* rt_dn, int* meta, int* ids_out,
                                 float* w_out, int* counts_out, cudaStream_t st);
// Large batches: routing plus per-block expert histograms (blockhist, zero
// at launch), scanned by the last CTA into counts, offsets, row tiles and
// per-block bases; then the stable scatter of the slots, in the same launch
// as the shared-expert gate logits.
cudaError_t launch_route_count(int T, int E, int k, int score_fn, int bn_gu, int bn_dn,
                               const LogitSrc& logits, bool pdl, int* topk_ids, float* topk_w,
                               int* blockhist, int* counts, int* offsets, int4* rt_gu, int4* rt_dn,
                               int* meta, int* ids_out, float* w_out, int* counts_out,
                               cudaStream_t st);
cudaError_t launch_scatter(int T, int H, int E, int k, const int* topk_ids, const int* blockhist,
                           const int* offsets, int* perm, int* inv, const __nv_bfloat16* hidden,
                           const __nv_bfloat16* w_g, float* gate_logit, cudaStream_t st);
// y: fp32 rows [T*k + T, H], or with `y16` the codes and exponent plane of
// the y16 format starting at y.
cudaError_t launch_combine(int T, int H, int k, const float* y, bool y16, const float* topk_w,
                           const int* inv, __nv_bfloat16* out, cudaStream_t st);
// Expert parallelism: the fp32 combine with the routed rows y_routed [T*k, H]
// (sorted order) and the gated shared rows y_shared [T, H] in separate arrays;
// the hidden rows of the (token, slot) pairs in sorted order; the row tiles of
// the received rows (G source segments of E_loc local experts).
constexpr int kEpTileThreads = 1024;
cudaError_t launch_combine_split(int T, int H, int k, const float* y_routed, const float* y_shared,
                                 const float* topk_w, const int* inv, __nv_bfloat16* out,
                                 cudaStream_t st);
cudaError_t launch_gather_rows(int P, int H, int k, const int* perm,
                               const __nv_bfloat16* hidden, __nv_bfloat16* rows, cudaStream_t st);
cudaError_t launch_ep_tiles(int G, int E_loc, int R, const int* recv_counts, int bn_gu,
                            int bn_dn, int4* rt_gu, int4* rt_dn, int* meta, cudaStream_t st);

// Grouped GEMMs (moe_gemm.cu).
struct GemmArgs {
    int T, H, E, k, I, I_s;
    int P;                  // routed rows (T*k; the received rows with expert parallelism)
    const __nv_bfloat16* hidden;
    // Routed rows already gathered in sorted order (row p = xrows[p]), or null:
    // row p is hidden[perm[p] / k]. Shared-expert rows always come from hidden.
    const __nv_bfloat16* xrows;
    const int* perm;
    const int* counts;
    const int* offsets;
    const int4* rowtiles;   // routed row tiles {expert, first row, rows, sorted position}
    const int* meta;
    int* sched;             // this GEMM's tile-claim counter (zero at launch)
    const float* gate_logit;
    __nv_bfloat16* h_hi;
    __nv_bfloat16* h_lo;
    __nv_bfloat16* hs_hi;
    __nv_bfloat16* hs_lo;
    float* y;
    uint8_t* yexp;          // y16 exponent plane (tokens-on-M down tiles)
    // routed y rows from this one on are stored with an L2 evict-last policy
    // (the rows written last, which the combine can then read from L2)
    int y_keep_row;
    unsigned* err;
    // NVFP4 weights: fp32 matrix scales of this GEMM's routed experts [E] and
    // of the shared expert [1]; null for bf16 and MXFP8 weights.
    const float* msc;
    const float* msc_s;
    // gate_up (bf16): the routed gate/up weights [E, 2I, H], read only by an
    // L2 prefetch issued before the wait for routing (null: no prefetch).
    const __nv_bfloat16* w_gu;
};

struct GemmMaps {
    // Operand loads (128-byte swizzle). A TMA request costs about the same
    // time whatever its size, so pairs of tiles that are always loaded
    // together come from one 3D box whose outer dimension (2) selects the
    // member of the pair; the box lands as two consecutive tiles.
    // gate_up: w / ws = W_gate_up as [E*2I - I rows, H] x {gate, up} (plane
    //   stride I rows), Ws_gate_up as [I_s, H] x {gate, up}; boxes 64 x NF x 2
    //   (NF = gate_up_ts_features(BN) gate and up rows per tile).
    // down: w / ws = W_down as [E*H, I] and Ws_down as [H, I_s]; h / hs = the
    //   h_hi and h_lo planes of [T*k, I] and [T, I_s]. 128-token tiles: 2D
    //   weight boxes of 64 x 256 rows and h boxes 64 x 128 x 2; the fused
    //   expert launch: 64 x 128 and 64 x BN x 2; down_kernel: the same boxes
    //   with kDownChunks 64-column chunks per request (an outer dimension of
    //   64-column chunks, 128-byte stride).
    CUtensorMap w;
    CUtensorMap ws;
    CUtensorMap h;
    CUtensorMap hs;
    // Epilogue stores of the down GEMM: st[0] = y [T*k + T, H] fp32 in boxes of
    // 32 columns x kEpiRows rows (no swizzle); with tokens on M, st[1] = the
    // y16 codes of y in boxes of 64 bytes x 32 rows. (The gate_up epilogues
    // write h with plain stores.)
    CUtensorMap st[4];
};

// TMA maps of the GEMMs with block-quantised expert weights (moe_gemm_mx.cu),
// listed for MXFP8; NVFP4 differs in the code and scale maps only: gate_up
// codes {H/2 bytes, rows, 2} in boxes 64 x 128 x 2 with the 64-byte swizzle,
// scales (E4M3, one per 16 values) {I, 2, E*H/16} in boxes 128 x 2 x 8; down
// codes {I/2 bytes, E*H rows} in boxes 128 x 128, scales {H, E*I/16} in boxes
// 128 x 16. Codes are bytes read with the 128-byte swizzle, scales bytes
// without swizzle.
// gate_up: w / ws = codes of W_gate_up as {H, E*2I - I rows, 2} (plane
//   stride I rows: gate, up) and of Ws_gate_up as {H, I_s, 2}, boxes
//   128 x 128 x 2; sc / scs = their scales [E, H/32, 2I] as {I, 2, E*H/32}
//   and [H/32, 2I_s] as {I_s, 2, H/32}, boxes 128 x 2 x 4.
// down: w / ws = codes of W_down as {128, I/128, E*H rows} and of Ws_down as
//   {128, I_s/128, H}, boxes 128 x 2 x 128 (256 K values of 128 rows, each
//   row's two 128-byte halves adjacent); sc / scs = scales [E, I/32, H] as
//   {H, E*I/32} and [I_s/32, H] as {H, I_s/32}, boxes 128 x 8; h / hs = h in
//   64-column panels (below) as {64, P rows, 2 (hi, lo), I/64 panels}, boxes
//   64 x BN x 2 x 4.
// h of the MXFP8 path is stored in 64-column panels: panel c holds columns
//   64c..64c+63 of the P rows of h_hi, then of h_lo (P = T*k routed, T
//   shared), so one box brings the hi and lo rows of four 64-column K
//   slices (the gate_up epilogue writes the panels with plain stores).
//   st[0] (down) = y.
struct MxMaps {
    CUtensorMap w;
    CUtensorMap ws;
    CUtensorMap sc;
    CUtensorMap scs;
    CUtensorMap h;
    CUtensorMap hs;
    CUtensorMap st[4];
};

// Supported tile widths (tokens per tile) of both GEMMs.
bool gemm_bn_supported(int bn);
cudaError_t launch_gate_up(int bn, const GemmMaps& maps, const GemmArgs& a, int max_tiles,
                           int num_sms, cudaStream_t st);
// One CTA that waits on an mbarrier nothing arrives on (bounded wait self-test).
cudaError_t launch_wait_limit_selftest(unsigned* err, cudaStream_t st);
cudaError_t launch_down(int bn, const GemmMaps& maps, const GemmArgs& a, int max_tiles,
                        int num_sms, cudaStream_t st);

// GEMMs with block-quantised weights (moe_gemm_mx.cu): MXFP8, or NVFP4 with
// `nvfp4`; tile widths 16, 32 and 64; H, I and I_s multiples of 128.
bool gemm_mx_bn_supported(int bn);
cudaError_t launch_gate_up_mx(int bn, bool nvfp4, const MxMaps& maps, const GemmArgs& a,
                              int max_tiles, int num_sms, cudaStream_t st);
cudaError_t launch_down_mx(int bn, bool nvfp4, const MxMaps& maps, const GemmArgs& a,
                           int max_tiles, int num_sms, cudaStream_t st);
// bf16 values (without the matrix scale) of an NVFP4 matrix [rows, cols]:
// codes [rows, cols/2], scales [cols/16, rows].
cudaError_t launch_nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, int rows, int cols,
                                 __nv_bfloat16* out, cudaStream_t st);
// Router GEMM (moe_router.cu): logits [T, E] fp32 = hidden [T, H] . W_router [E, H]^T,
// as a split-K GEMM (tiles of 128 experts x bn tokens, `splits` K ranges) that
// writes the partial sums [splits, T, E]; the routing kernels add them in a
// fixed order (LogitSrc).
constexpr int kRouterMaxSplits = 32;
struct RouterPlan {
    int bn;      // tokens per tile (16 .. 256)
    int splits;  // K ranges (1 = the GEMM writes the logits directly)
};
int router_max_splits(int T, int H, int E);  // bound on splits (sizes the workspace)
RouterPlan router_plan(int T, int H, int E, int num_sms);
// map_w: W_router [E, H] in boxes of 64 x 128 rows; map_x: hidden [T, H], boxes 64 x bn.
cudaError_t launch_router(const RouterPlan& p, const CUtensorMap& map_w, const CUtensorMap& map_x,
                          int T, int H, int E, float* partial, unsigned* err, cudaStream_t st);

// bf16 values of an MXFP8 matrix [rows, cols] (scales [cols/32, rows]).
cudaError_t launch_mxfp8_dequant(const uint8_t* codes, const uint8_t* scales, int rows, int cols,
                                 __nv_bfloat16* out, cudaStream_t st);

}  // namespace moe
