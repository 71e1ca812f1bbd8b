// C ABI of libmoe: argument checks, workspace carving, TMA descriptors and
// the launch sequence route (+ histogram/scan) -> scatter -> gate_up -> down
// -> combine on the caller's stream. See include/moe.h for the contract.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "moe.h"
#include "moe_fused.cuh"
#include "moe_internal.cuh"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {
namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxDevices = 64;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
    size_t meta, ready, topk_ids, topk_w, gate_logit, counts, offsets, perm, inv, blockhist;
    size_t rt_gu, rt_dn, h_hi, h_lo, hs_hi, hs_lo, y, total;
};

bool dims_valid(const moe_dims* d) {
    if (!d) return false;
    if (d->T < 0 || d->T > (1 << 22)) return false;
    if (d->E < 1 || d->E > 1024) return false;
    if (d->k < 1 || d->k > 32 || d->k > d->E) return false;
    if (d->H < 1 || d->H > 65536 || d->I < 1 || d->I > 65536 || d->I_s < 1 || d->I_s > 65536)
        return false;
    if (d->score_fn != MOE_SCORE_SOFTMAX && d->score_fn != MOE_SCORE_SIGMOID) return false;
    return true;
}

bool dims_supported(const moe_dims* d) {
    return d->H % 64 == 0 && d->I % 64 == 0 && d->I_s % 64 == 0 && d->H >= 64 && d->I >= 64 &&
           d->I_s >= 64;
}

// Upper bound on the routed row tiles of a GEMM with tile width bn.
size_t max_row_tiles(size_t tk, size_t E, size_t bn) { return tk / bn + (tk < E ? tk : E) + 1; }

Layout layout_of(const moe_dims& d) {
    Layout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + (bytes ? bytes : 1), kAlign);
        return o;
    };
    const size_t T = d.T, H = d.H, E = d.E, I = d.I, Is = d.I_s, tk = T * d.k;
    const size_t nb = (T + kCountTokens - 1) / kCountTokens;
    // The status block, the large-batch routing's block histograms and the
    // fused launch's readiness counters are adjacent: one memset clears what
    // a call needs of them.
    L.meta = take(META_WORDS * sizeof(int));
    L.blockhist = take(nb * E * 4);
    L.ready = take((tk + T) * 4);
    L.topk_ids = take(tk * 4);
    L.topk_w = take(tk * 4);
    L.gate_logit = take(T * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.perm = take(tk * 4);
    L.inv = take(tk * 4);
    L.rt_gu = take(max_row_tiles(tk, E, 16) * sizeof(int4));
    L.rt_dn = take(max_row_tiles(tk, E, 16) * sizeof(int4));
    L.h_hi = take(tk * I * 2);
    L.h_lo = take(tk * I * 2);
    L.hs_hi = take(T * Is * 2);
    L.hs_lo = take(T * Is * 2);
    L.y = take((tk + T) * H * 4);
    L.total = off;
    return L;
}

// Extra workspace of the FFN-side router, after the standard layout: the
// router GEMM's split-K partial sums [max splits, T, E] fp32.
struct RouterLayout {
    size_t partial, total;
};

RouterLayout router_layout_of(const moe_dims& d) {
    RouterLayout R{};
    const size_t n = static_cast<size_t>(d.T) * d.E;
    const int cap = router_max_splits(d.T, d.H, d.E);
    R.partial = layout_of(d).total;
    R.total = align_up(R.partial + (n ? static_cast<size_t>(cap) * n * 4 : 1), kAlign);
    return R;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Row-major bf16 matrix [outer, inner] read in boxes of 64 x box_rows with
// the 128-byte swizzle; out-of-range rows read as zero.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kGemmBK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Pair of bf16 matrices [rows, inner], the second `plane_bytes` after the
// first, as one 3D map {inner, rows, 2}; a box of 64 x box_rows x 2 lands as
// the first matrix's rows followed by the second's (128-byte swizzle).
bool make_pair_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                   uint64_t plane_bytes, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {inner, rows, 2};
    cuuint64_t strides[2] = {inner * 2, plane_bytes};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kGemmBK), box_rows, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major bf16 matrix [rows, inner] (inner a multiple of 64) viewed as
// {64, rows, inner / 64}: a box of 64 x box_rows x kc lands as kc consecutive
// 64-column chunks of box_rows rows each (128-byte swizzle), the layout of kc
// separate 2D boxes in one request; chunks past `inner` read as zero.
bool make_chunk_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                    uint32_t box_rows, uint32_t kc) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kGemmBK), rows, inner / kGemmBK};
    cuuint64_t strides[2] = {inner * 2, static_cast<cuuint64_t>(kGemmBK) * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kGemmBK), box_rows, kc};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The pair map above (two matrices [rows, inner], `plane_bytes` apart) viewed
// as {64, rows, 2, inner / 64}: a box of 64 x box_rows x 2 x kc lands as kc
// chunks, each the first matrix's rows then the second's.
bool make_pair_chunk_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                         uint64_t plane_bytes, uint32_t box_rows, uint32_t kc) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(kGemmBK), rows, 2, inner / kGemmBK};
    cuuint64_t strides[3] = {inner * 2, plane_bytes, static_cast<cuuint64_t>(kGemmBK) * 2};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(kGemmBK), box_rows, 2, kc};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Operand maps of the bf16 down GEMM (GemmMaps w, ws, h, hs): W_down [E*H, I],
// Ws_down [H, I_s] and the h_hi / h_lo planes of [P, I] and [T, I_s]. The
// tokens-on-M kernels (128-token tiles; stacked 64-token tiles) read 256
// weight rows per request; the fused expert launch 64-K steps; down_kernel
// kDownChunks 64-K chunks per request.
bool make_down_maps(GemmMaps* dn, const void* w_down, const void* ws_down, const void* h_hi,
                    const void* hs_hi, uint64_t h_plane, uint64_t hs_plane, uint64_t E, uint64_t H,
                    uint64_t I, uint64_t Is, uint64_t T, uint64_t P, int bn_dn, bool fused) {
    const uint32_t bn = static_cast<uint32_t>(bn_dn);
    if (bn_dn >= 64 || fused) {
        // 128-token and stacked 64-token tiles: 256 weight rows per request
        const uint32_t w_rows = (!fused && bn_dn >= 64) ? 256u : static_cast<uint32_t>(kGemmBM);
        return make_map(&dn->w, w_down, I, E * H, w_rows) &&
               make_map(&dn->ws, ws_down, Is, H, w_rows) &&
               make_pair_map(&dn->h, h_hi, I, P, h_plane, bn) &&
               make_pair_map(&dn->hs, hs_hi, Is, T, hs_plane, bn);
    }
    const uint32_t kc = kDownChunks;
    return make_chunk_map(&dn->w, w_down, I, E * H, kGemmBM, kc) &&
           make_chunk_map(&dn->ws, ws_down, Is, H, kGemmBM, kc) &&
           make_pair_chunk_map(&dn->h, h_hi, I, P, h_plane, bn, kc) &&
           make_pair_chunk_map(&dn->hs, hs_hi, Is, T, hs_plane, bn, kc);
}

// Tiled map of `rank` dimensions over bytes (dt UINT8) or bf16; dims and box
// innermost first, strides[i] = byte stride of dimension i + 1.
bool make_map_nd(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int rank,
                 const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                 CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], estr[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        estr[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    return fn(m, dt, rank, const_cast<void*>(base), d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swz, swz == CU_TENSOR_MAP_SWIZZLE_NONE ? CU_TENSOR_MAP_L2_PROMOTION_NONE
                                                     : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major matrix [outer, inner] of `elem` bytes per element, written by the
// GEMM epilogues in boxes of kEpiCols x kEpiRows (no swizzle).
bool make_store_map(CUtensorMap* m, void* base, CUtensorMapDataType dt, uint32_t elem,
                    uint64_t inner, uint64_t outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * elem};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kEpiCols), static_cast<cuuint32_t>(kEpiRows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// y16 codes of y (rows of 2H bytes, byte tensor [outer, 2 * inner]) written
// in boxes of 64 bytes (32 values) x box_rows rows.
bool make_y16_store_map(CUtensorMap* m, void* base, uint64_t inner, uint64_t outer,
                        uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {2 * inner, outer};
    cuuint64_t strides[1] = {2 * inner};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Bytes of y16 rows the tokens-on-M down GEMM stores with an L2 evict-last
// policy (the last routed rows it writes), for the combine to read from L2.
constexpr size_t kYKeepBytes = size_t(64) << 20;

int sm_count() {
    static int cache[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= kMaxDevices) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

// Tokens per tile: the smallest supported width >= 1.25x the mean group size.
// gate_up also has a 160-token width (groups of ~128 tokens fit one tile and
// the pipeline keeps four stages).
int pick_bn(size_t tk, int E, int cap, bool gate_up) {
    const double mean = static_cast<double>(tk) / E;
    const int widths[] = {16, 32, 64, 128, 160, 256};
    int bn = 16;
    for (int w : widths) {
        if (w > cap || (w == 160 && !gate_up)) continue;
        bn = w;
        if (w >= 1.25 * mean) break;
    }
    return bn;
}

// Per host thread: may moe_forward / moe_forward_router fuse launches
// (moe_set_expert_fusion)? 0 (default): no; 1: gate_up and down as one
// launch; 2: also the whole layer in one launch where it applies. Off by
// default: measured on GB300, the fused launches are no faster at decode (the
// programmatic dependent launches already overlap the boundaries) and the
// fused expert launch is slower on wide batches (its down steps share the
// gate_up-sized ring and keep fewer bytes in flight).
thread_local int tl_fusion = 0;

// Token-tile widths of the two bf16 GEMMs, and which launches are fused.
struct BnPlan {
    int gu, dn;
    bool fused;  // gate_up and down in one launch
    bool layer;  // routing, both GEMMs and the combine in one launch
};

BnPlan bn_plan(size_t tk, int E, bool mx, bool router = false) {
    BnPlan p;
    p.gu = pick_bn(tk, E, mx ? 64 : 256, true);
    p.dn = pick_bn(tk, E, mx ? 64 : 128, false);
    p.fused = !mx && tl_fusion >= 1 && p.gu == p.dn && p.gu <= kFusedMaxBN;
    p.layer = p.fused && tl_fusion >= 2 && !router && tk <= static_cast<size_t>(kSmallSlots) &&
              E <= kLayerMaxExperts;
    return p;
}

// Kernels one forward launches: routing (one launch, or route with the block
// histograms + scatter), the expert GEMMs (one fused launch or two), the
// combine; or the whole layer as one launch.
int launches_of(const moe_dims& d, bool mx, bool router = false) {
    const size_t tk = static_cast<size_t>(d.T) * d.k;
    const BnPlan p = bn_plan(tk, d.E, mx, router);
    if (p.layer) return 1;
    return (route_small_fits(d.T, d.E, d.k) ? 1 : 2) + (p.fused ? 1 : 2) + 1;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Caller-owned timing events of this host thread (moe_set_stage_events).
thread_local cudaEvent_t tl_stage_events[MOE_NUM_STAGES + 1];
thread_local bool tl_stage_events_on = false;

void mark_stage(int i, cudaStream_t st) {
    if (tl_stage_events_on) cudaEventRecord(tl_stage_events[i], st);
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API size_t moe_workspace_size(const moe_dims* d) {
    if (!dims_valid(d)) return 0;
    return layout_of(*d).total;
}

MOE_API moe_status moe_workspace_layout(const moe_dims* d, moe_workspace_layout_t* out) {
    if (!dims_valid(d) || !out) return MOE_ERR_INVALID_ARG;
    const Layout L = layout_of(*d);
    out->topk_ids = L.topk_ids;
    out->topk_w = L.topk_w;
    out->gate_logit = L.gate_logit;
    out->counts = L.counts;
    out->offsets = L.offsets;
    out->perm = L.perm;
    out->inv = L.inv;
    out->h_hi = L.h_hi;
    out->h_lo = L.h_lo;
    out->hs_hi = L.hs_hi;
    out->hs_lo = L.hs_lo;
    out->y = L.y;
    out->total = L.total;
    return MOE_OK;
}

MOE_API const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED:
            return "unsupported size (H, I and I_s must be multiples of 64; of 128 for MXFP8 or "
                   "NVFP4 weights)";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
        case MOE_ERR_CAPACITY: return "sizes exceed the fixed static scratch (ceil(T/256)*E > 2^18)";
        default: return "unknown status";
    }
}

namespace moe {
namespace {

// The experts' weights: bf16 matrices, or block-quantised codes with their
// scales (mx: MXFP8, or NVFP4 when nv is also set).
struct ExpertWeights {
    bool mx;
    bool nv;
    const void* gate_up;      // [E, 2I, H] bf16, E4M3 codes, or [E, 2I, H/2] E2M1 pairs
    const void* down;         // [E, H, I] (NVFP4: [E, H, I/2])
    const void* s_gate_up;    // shared expert [2I_s, H]
    const void* s_down;       // shared expert [H, I_s]
    const uint8_t* gate_up_sc;    // block scales [E, H/B, 2I] (B = 32 MXFP8, 16 NVFP4)
    const uint8_t* down_sc;       // [E, I/B, H]
    const uint8_t* s_gate_up_sc;  // [H/B, 2I_s]
    const uint8_t* s_down_sc;     // [I_s/B, H]
    const float* g_gate_up;       // NVFP4 matrix scales [E]
    const float* g_down;          // [E]
    const float* g_s_gate_up;     // [1]
    const float* g_s_down;        // [1]
};

bool dims_supported_mx(const moe_dims* d) {
    return d->H % 128 == 0 && d->I % 128 == 0 && d->I_s % 128 == 0;
}

// TMA maps of the block-quantised GEMMs (layouts in moe_internal.cuh, MxMaps).
bool make_mx_maps(const moe_dims& d, const ExpertWeights& W, const Layout& L, char* ws, int bn_dn,
                  MxMaps* gu, MxMaps* dn) {
    const uint64_t T = d.T, H = d.H, E = d.E, I = d.I, Is = d.I_s, tk = T * d.k;
    const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const CUtensorMapDataType BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapSwizzle SW = CU_TENSOR_MAP_SWIZZLE_128B, NOSW = CU_TENSOR_MAP_SWIZZLE_NONE;
    bool ok = true;
    const uint64_t B = W.nv ? 16 : 32;  // K values per block scale
    {   // gate_up codes: {row bytes, rows, 2 (gate, up)}: MXFP8 boxes 128 x 128 x 2
        // (128 K), NVFP4 boxes 64 x 128 x 2 (128 K at half a byte, 64-byte swizzle)
        const uint64_t rb = W.nv ? H / 2 : H;
        const uint32_t box[3] = {W.nv ? 64u : 128u, 128, 2};
        const CUtensorMapSwizzle sz = W.nv ? CU_TENSOR_MAP_SWIZZLE_64B : SW;
        const uint64_t dw[3] = {rb, E * 2 * I - I, 2}, sw[2] = {rb, I * rb};
        const uint64_t ds[3] = {rb, Is, 2}, ss[2] = {rb, Is * rb};
        ok = ok && make_map_nd(&gu->w, U8, W.gate_up, 3, dw, sw, box, sz) &&
             make_map_nd(&gu->ws, U8, W.s_gate_up, 3, ds, ss, box, sz);
    }
    {   // gate_up scales: {rows of a plane, 2 planes, K blocks}, boxes 128 x 2 x (128 / B)
        const uint32_t box[3] = {128, 2, static_cast<uint32_t>(128 / B)};
        const uint64_t dw[3] = {I, 2, E * (H / B)}, sw[2] = {I, 2 * I};
        const uint64_t ds[3] = {Is, 2, H / B}, ss[2] = {Is, 2 * Is};
        ok = ok && make_map_nd(&gu->sc, U8, W.gate_up_sc, 3, dw, sw, box, NOSW) &&
             make_map_nd(&gu->scs, U8, W.s_gate_up_sc, 3, ds, ss, box, NOSW);
    }
    if (W.nv) {  // down codes: {I/2 bytes, rows}, boxes 128 x 128 (256 K values)
        const uint32_t box[2] = {128, 128};
        const uint64_t dw[2] = {I / 2, E * H}, sw[1] = {I / 2};
        const uint64_t ds[2] = {Is / 2, H}, ss[1] = {Is / 2};
        ok = ok && make_map_nd(&dn->w, U8, W.down, 2, dw, sw, box, SW) &&
             make_map_nd(&dn->ws, U8, W.s_down, 2, ds, ss, box, SW);
    } else {  // down codes: {128, K / 128, rows}, boxes 128 x 2 x 128
        const uint32_t box[3] = {128, 2, 128};
        const uint64_t dw[3] = {128, I / 128, E * H}, sw[2] = {128, I};
        const uint64_t ds[3] = {128, Is / 128, H}, ss[2] = {128, Is};
        ok = ok && make_map_nd(&dn->w, U8, W.down, 3, dw, sw, box, SW) &&
             make_map_nd(&dn->ws, U8, W.s_down, 3, ds, ss, box, SW);
    }
    {   // down scales: {H, K blocks}, boxes 128 x (256 / B)
        const uint32_t box[2] = {128, static_cast<uint32_t>(256 / B)};
        const uint64_t dw[2] = {H, E * (I / B)}, sw[1] = {H};
        const uint64_t ds[2] = {H, Is / B}, ss[1] = {H};
        ok = ok && make_map_nd(&dn->sc, U8, W.down_sc, 2, dw, sw, box, NOSW) &&
             make_map_nd(&dn->scs, U8, W.s_down_sc, 2, ds, ss, box, NOSW);
    }
    {   // h panels: {64, P, 2 (hi, lo), K / 64}, boxes 64 x BN x 2 x 4
        const uint32_t box[4] = {64, static_cast<uint32_t>(bn_dn), 2, 4};
        const uint64_t dr[4] = {64, tk, 2, I / 64}, sr[3] = {128, tk * 128, 2 * tk * 128};
        const uint64_t dsh[4] = {64, T, 2, Is / 64}, ssh[3] = {128, T * 128, 2 * T * 128};
        ok = ok && make_map_nd(&dn->h, BF16, ws + L.h_hi, 4, dr, sr, box, SW) &&
             make_map_nd(&dn->hs, BF16, ws + L.hs_hi, 4, dsh, ssh, box, SW);
    }
    ok = ok && make_store_map(&dn->st[0], ws + L.y, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, tk + T) &&
         make_y16_store_map(&dn->st[2], ws + L.y, H, tk + T, kEpiRows);
    return ok;
}

// Device arrays the routing and permute kernels write.
struct RouteBufs {
    int* topk_ids;
    float* topk_w;
    float* gate_logit;
    int* blockhist;
    int* counts;
    int* offsets;
    int* perm;
    int* inv;
    int4* rt_gu;
    int4* rt_dn;
    int* meta;
};

// Routing and the permute (stage 0, and the scatter as stage 1): one launch
// when T*k <= 2048, else routing with the block histograms, then the scatter
// (whose launch also computes the gate logits). The status words (and, for large batches, the block histograms) must be
// zero.
cudaError_t enqueue_routing(int T, int H, int E, int k, int score_fn, int bn_gu, int bn_dn,
                            const LogitSrc& lsrc, bool pdl, const void* hidden, const void* w_g,
                            const RouteBufs& b, int* ids_out, float* w_out, int* counts_out,
                            cudaStream_t st) {
    const auto* x = static_cast<const __nv_bfloat16*>(hidden);
    const auto* g = static_cast<const __nv_bfloat16*>(w_g);
    cudaError_t e;
    if (route_small_fits(T, E, k)) {
        e = launch_route_permute(T, H, E, k, score_fn, bn_gu, bn_dn, lsrc, pdl, x, g, b.topk_ids,
                                 b.topk_w, b.gate_logit, b.counts, b.offsets, b.perm, b.inv,
                                 b.rt_gu, b.rt_dn, b.meta, ids_out, w_out, counts_out, st);
        mark_stage(1, st);
        return e;
    }
    e = launch_route_count(T, E, k, score_fn, bn_gu, bn_dn, lsrc, pdl, b.topk_ids, b.topk_w,
                           b.blockhist, b.counts, b.offsets, b.rt_gu, b.rt_dn, b.meta, ids_out,
                           w_out, counts_out, st);
    if (e != cudaSuccess) return e;
    mark_stage(1, st);
    return launch_scatter(T, H, E, k, b.topk_ids, b.blockhist, b.offsets, b.perm, b.inv, x, g,
                          b.gate_logit, st);
}

// Bytes of the status block (and the block histograms of large batches) a
// call must clear before routing T tokens; the histograms follow the status
// block in every workspace layout.
size_t routing_zero_bytes(const Layout& L, int T, int E, int k) {
    if (route_small_fits(T, E, k)) return META_WORDS * sizeof(int);
    return L.blockhist - L.meta +
           static_cast<size_t>((T + kCountTokens - 1) / kCountTokens) * E * sizeof(int);
}

// w_router == nullptr: router_logits are an input. Otherwise the layer first
// computes them from w_router [E, H] into logits_out (if given) or its
// workspace (router_logits must then be null).
moe_status forward_impl(const moe_dims* d, const void* hidden, const float* router_logits,
                        const void* w_router, float* logits_out, const ExpertWeights& W,
                        const void* w_g, void* out, int32_t* topk_ids_out, float* topk_w_out,
                        int32_t* expert_counts_out, void* workspace, size_t workspace_bytes,
                        void* cuda_stream) {
    if (!dims_valid(d)) return MOE_ERR_INVALID_ARG;
    if (!dims_supported(d) || (W.mx && !dims_supported_mx(d))) return MOE_ERR_UNSUPPORTED;
    if (d->T == 0) return MOE_OK;
    if (w_router) {
        if (router_logits) return MOE_ERR_INVALID_ARG;
        if (!aligned16(w_router) || (logits_out && !aligned16(logits_out)))
            return MOE_ERR_INVALID_ARG;
    }
    const void* required[] = {hidden, w_router ? w_router : router_logits, W.gate_up, W.down,
                              W.s_gate_up, W.s_down, w_g, out};
    for (const void* p : required)
        if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (W.mx) {
        const void* scales[] = {W.gate_up_sc, W.down_sc, W.s_gate_up_sc, W.s_down_sc};
        for (const void* p : scales)
            if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    }
    if (W.nv) {
        const void* gs[] = {W.g_gate_up, W.g_down, W.g_s_gate_up, W.g_s_down};
        for (const void* p : gs)
            if (!p || (reinterpret_cast<uintptr_t>(p) & 3u)) return MOE_ERR_INVALID_ARG;
    }
    const void* optional[] = {topk_ids_out, topk_w_out, expert_counts_out};
    for (const void* p : optional)
        if (p && (reinterpret_cast<uintptr_t>(p) & 3u)) return MOE_ERR_INVALID_ARG;
    const Layout L = layout_of(*d);
    const RouterLayout RL = router_layout_of(*d);
    if (!workspace || workspace_bytes < (w_router ? RL.total : L.total) ||
        (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
        return MOE_ERR_WORKSPACE;

    const int T = d->T, H = d->H, E = d->E, k = d->k, I = d->I, Is = d->I_s;
    const size_t tk = static_cast<size_t>(T) * k;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    char* ws = static_cast<char*>(workspace);
    int* meta = reinterpret_cast<int*>(ws + L.meta);
    int* topk_ids = reinterpret_cast<int*>(ws + L.topk_ids);
    float* topk_w = reinterpret_cast<float*>(ws + L.topk_w);
    float* gate_logit = reinterpret_cast<float*>(ws + L.gate_logit);
    int* counts = reinterpret_cast<int*>(ws + L.counts);
    int* offsets = reinterpret_cast<int*>(ws + L.offsets);
    int* perm = reinterpret_cast<int*>(ws + L.perm);
    int* inv = reinterpret_cast<int*>(ws + L.inv);
    int* blockhist = reinterpret_cast<int*>(ws + L.blockhist);
    int4* rt_gu = reinterpret_cast<int4*>(ws + L.rt_gu);
    int4* rt_dn = reinterpret_cast<int4*>(ws + L.rt_dn);
    auto* h_hi = reinterpret_cast<__nv_bfloat16*>(ws + L.h_hi);
    auto* h_lo = reinterpret_cast<__nv_bfloat16*>(ws + L.h_lo);
    auto* hs_hi = reinterpret_cast<__nv_bfloat16*>(ws + L.hs_hi);
    auto* hs_lo = reinterpret_cast<__nv_bfloat16*>(ws + L.hs_lo);
    float* y = reinterpret_cast<float*>(ws + L.y);

    // The MXFP8 GEMMs keep the weights on the MMA's M side at every size and
    // take tiles of at most 64 tokens.
    const BnPlan plan = bn_plan(tk, E, W.mx, w_router != nullptr);
    const int bn_gu = plan.gu, bn_dn = plan.dn;
    const int num_sms = sm_count();
    if (num_sms <= 0) return MOE_ERR_CUDA;

    GemmMaps gu{}, dn{};
    MxMaps mgu{}, mdn{};
    bool ok;
    if (W.mx) {
        ok = make_mx_maps(*d, W, L, ws, bn_dn, &mgu, &mdn);
    } else {
        // gate_up: the gate rows of expert e are rows e*2I + [0, I) of W_gate_up and its up
        // rows follow I rows later, so a map over the first E*2I - I rows with a plane stride
        // of I rows reaches both (and no address past the tensor); likewise I_s for the
        // shared expert. down: 128-token tiles read 256 weight rows per request.
        // (the tokens-on-M gate_up kernel reads gu_rows gate and up rows per tile)
        const uint32_t gu_rows = plan.fused ? static_cast<uint32_t>(kGemmBM)
                                            : static_cast<uint32_t>(gate_up_ts_features(bn_gu));
        ok = make_pair_map(&gu.w, W.gate_up, H, static_cast<uint64_t>(E) * 2 * I - I,
                           static_cast<uint64_t>(I) * H * 2, gu_rows) &&
             make_pair_map(&gu.ws, W.s_gate_up, H, Is, static_cast<uint64_t>(Is) * H * 2,
                           gu_rows) &&
             make_down_maps(&dn, W.down, W.s_down, h_hi, hs_hi, L.h_lo - L.h_hi,
                            L.hs_lo - L.hs_hi, E, H, I, Is, T, tk, bn_dn, plan.fused);
        ok = ok && make_store_map(&dn.st[0], y, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, tk + T) &&
             make_y16_store_map(&dn.st[1], y, H, tk + T, 32) &&
             make_y16_store_map(&dn.st[2], y, H, tk + T, kEpiRows);
    }
    if (!ok) return MOE_ERR_CUDA;

    GemmArgs ga{};
    ga.T = T;
    ga.H = H;
    ga.E = E;
    ga.k = k;
    ga.I = I;
    ga.I_s = Is;
    ga.P = static_cast<int>(tk);
    ga.hidden = static_cast<const __nv_bfloat16*>(hidden);
    ga.perm = perm;
    ga.counts = counts;
    ga.offsets = offsets;
    ga.meta = meta;
    ga.gate_logit = gate_logit;
    ga.h_hi = h_hi;
    ga.h_lo = h_lo;
    ga.hs_hi = hs_hi;
    ga.hs_lo = hs_lo;
    ga.y = y;
    // y as y16 codes (the exponent plane after them) where its bytes matter:
    // the tokens-on-M down tiles always, the others when fp32 y would exceed
    // 64 MB. Decode-sized batches keep fp32 y, whose combine has more threads
    // in flight per output.
    const bool y16 = (!W.mx && bn_dn == 128) || (tk + T) * static_cast<size_t>(H) * 4 > (64u << 20);
    if (y16) ga.yexp = reinterpret_cast<uint8_t*>(y) + (tk + T) * 2 * static_cast<size_t>(H);
    // The routed y rows written last (tiles are claimed in expert order) stay in
    // L2 for the combine, up to kYKeepBytes of them.
    {
        const size_t keep_rows = kYKeepBytes / (2 * static_cast<size_t>(H));
        ga.y_keep_row = static_cast<int>(tk > keep_rows ? tk - keep_rows : 0);
    }
    ga.err = reinterpret_cast<unsigned*>(meta + META_ERR);
    GemmArgs gd = ga;
    ga.rowtiles = rt_gu;
    gd.rowtiles = rt_dn;
    if (W.nv) {
        ga.msc = W.g_gate_up;
        ga.msc_s = W.g_s_gate_up;
        gd.msc = W.g_down;
        gd.msc_s = W.g_s_down;
    }
    ga.sched = meta + META_SCHED_GU;
    gd.sched = meta + META_SCHED_DN;
    // Decode-sized batches: L2 prefetch of the first tiles' weights while routing
    // finishes (measured: decode -1.8 us; wider tiles: no gain or slower).
    if (!W.mx && bn_gu <= 32) ga.w_gu = static_cast<const __nv_bfloat16*>(W.gate_up);

    const size_t routed_min = tk < static_cast<size_t>(E) ? tk : static_cast<size_t>(E);
    const int gu_nf = W.mx || plan.fused ? kGemmBM : gate_up_ts_features(bn_gu);
    const int F_gu = (I + gu_nf - 1) / gu_nf, F_s = (Is + gu_nf - 1) / gu_nf;
    // 128-token down tiles use the tokens-on-M kernel with 256 output features per tile.
    // 128-token and (unfused bf16) 64-token down tiles take 256 output features.
    const bool dn256 = bn_dn == 128 || (bn_dn == 64 && !plan.fused && !W.mx);
    const int F_dn = dn256 ? (H + 255) / 256 : (H + kGemmBM - 1) / kGemmBM;
    const size_t max_gu = (tk / bn_gu + routed_min) * F_gu + ((T + bn_gu - 1) / bn_gu) * F_s;
    const size_t max_dn = (tk / bn_dn + routed_min) * F_dn + ((T + bn_dn - 1) / bn_dn) * F_dn;
    const int cap = 1 << 30;
    const int tiles_gu = static_cast<int>(max_gu < cap ? max_gu : cap);
    const int tiles_dn = static_cast<int>(max_dn < cap ? max_dn : cap);

    // Status words (error flags, tile counts, completion ticket) start at zero,
    // and so do the large-batch routing's block histograms and the fused
    // launch's row-tile readiness counters that follow them.
    const size_t zero_bytes = plan.fused ? L.ready - L.meta + (tk + T) * sizeof(int)
                                         : routing_zero_bytes(L, T, E, k);
    if (cudaMemsetAsync(meta, 0, zero_bytes, st) != cudaSuccess) return MOE_ERR_CUDA;
    mark_stage(0, st);
    LogitSrc lsrc{router_logits, 1, 0, nullptr};
    if (w_router) {
        // The router GEMM belongs to stage 0; the routing kernels add its partial sums.
        const RouterPlan rp = router_plan(T, H, E, num_sms);
        CUtensorMap map_w{}, map_x{};
        if (!make_map(&map_w, w_router, H, E, kGemmBM) ||
            !make_map(&map_x, hidden, H, T, static_cast<uint32_t>(rp.bn)))
            return MOE_ERR_CUDA;
        float* partial = reinterpret_cast<float*>(ws + RL.partial);
        if (launch_router(rp, map_w, map_x, T, H, E, partial,
                          reinterpret_cast<unsigned*>(meta + META_ERR), st) != cudaSuccess)
            return MOE_ERR_CUDA;
        lsrc = LogitSrc{partial, rp.splits, static_cast<size_t>(T) * E, logits_out};
    }
    if (plan.layer) {
        // The whole layer in one launch: its time is stage 0's, the others are empty.
        int* ready = reinterpret_cast<int*>(ws + L.ready);
        LayerArgs la{};
        la.score_fn = d->score_fn;
        la.bn_gu = bn_gu;
        la.bn_dn = bn_dn;
        la.logits = lsrc;
        la.w_g = static_cast<const __nv_bfloat16*>(w_g);
        la.topk_ids = topk_ids;
        la.topk_w = topk_w;
        la.gate_logit = gate_logit;
        la.counts = counts;
        la.offsets = offsets;
        la.perm = perm;
        la.inv = inv;
        la.rt_gu = rt_gu;
        la.rt_dn = rt_dn;
        la.meta = meta;
        la.ids_out = topk_ids_out;
        la.w_out = topk_w_out;
        la.counts_out = expert_counts_out;
        la.out = static_cast<__nv_bfloat16*>(out);
        if (launch_layer_fused(bn_gu, gu, dn, ga, ready, la, num_sms, st) != cudaSuccess)
            return MOE_ERR_CUDA;
        for (int i = 1; i <= MOE_NUM_STAGES; ++i) mark_stage(i, st);
        return MOE_OK;
    }
    const RouteBufs rb{topk_ids, topk_w, gate_logit, blockhist, counts, offsets,
                       perm,     inv,    rt_gu,      rt_dn,     meta};
    if (enqueue_routing(T, H, E, k, d->score_fn, bn_gu, bn_dn, lsrc, w_router != nullptr, hidden,
                        w_g, rb, topk_ids_out, topk_w_out, expert_counts_out, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    mark_stage(2, st);
    if (plan.fused) {
        // gate_up and down in one launch; its time is stage 2's, stage 3 is empty.
        int* ready = reinterpret_cast<int*>(ws + L.ready);
        const int tiles = tiles_gu > cap - tiles_dn ? cap : tiles_gu + tiles_dn;
        if (launch_expert_fused(bn_gu, gu, dn, ga, ready, tiles, num_sms, st) != cudaSuccess)
            return MOE_ERR_CUDA;
        mark_stage(3, st);
        mark_stage(4, st);
    } else {
        const cudaError_t e_gu = W.mx ? launch_gate_up_mx(bn_gu, W.nv, mgu, ga, tiles_gu, num_sms, st)
                                      : launch_gate_up(bn_gu, gu, ga, tiles_gu, num_sms, st);
        if (e_gu != cudaSuccess) return MOE_ERR_CUDA;
        mark_stage(3, st);
        const cudaError_t e_dn = W.mx ? launch_down_mx(bn_dn, W.nv, mdn, gd, tiles_dn, num_sms, st)
                                      : launch_down(bn_dn, dn, gd, tiles_dn, num_sms, st);
        if (e_dn != cudaSuccess) return MOE_ERR_CUDA;
        mark_stage(4, st);
    }
    if ((launch_combine(T, H, k, y, y16, topk_w, inv,
                        static_cast<__nv_bfloat16*>(out), st)) != cudaSuccess)
        return MOE_ERR_CUDA;
    mark_stage(5, st);
    return MOE_OK;
}

}  // namespace
}  // namespace moe

MOE_API moe_status moe_forward(const moe_dims* d, const void* hidden, const float* router_logits,
                               const void* w_gate_up, const void* w_down, const void* ws_gate_up,
                               const void* ws_down, const void* w_g, void* out,
                               int32_t* topk_ids_out, float* topk_w_out,
                               int32_t* expert_counts_out, void* workspace,
                               size_t workspace_bytes, void* cuda_stream) {
    ExpertWeights W{};
    W.mx = false;
    W.gate_up = w_gate_up;
    W.down = w_down;
    W.s_gate_up = ws_gate_up;
    W.s_down = ws_down;
    return forward_impl(d, hidden, router_logits, nullptr, nullptr, W, w_g, out, topk_ids_out,
                        topk_w_out, expert_counts_out, workspace, workspace_bytes, cuda_stream);
}

MOE_API moe_status moe_forward_router(const moe_dims* d, const void* hidden, const void* w_router,
                                      const void* w_gate_up, const void* w_down,
                                      const void* ws_gate_up, const void* ws_down, const void* w_g,
                                      void* out, float* logits_out, int32_t* topk_ids_out,
                                      float* topk_w_out, int32_t* expert_counts_out,
                                      void* workspace, size_t workspace_bytes, void* cuda_stream) {
    if (!w_router) return MOE_ERR_INVALID_ARG;
    ExpertWeights W{};
    W.mx = false;
    W.gate_up = w_gate_up;
    W.down = w_down;
    W.s_gate_up = ws_gate_up;
    W.s_down = ws_down;
    return forward_impl(d, hidden, nullptr, w_router, logits_out, W, w_g, out, topk_ids_out,
                        topk_w_out, expert_counts_out, workspace, workspace_bytes, cuda_stream);
}

MOE_API size_t moe_workspace_size_router(const moe_dims* d) {
    if (!dims_valid(d)) return 0;
    return router_layout_of(*d).total;
}

MOE_API int moe_launch_count_router(const moe_dims* d) {
    if (!dims_valid(d) || !dims_supported(d) || d->T == 0) return 0;
    return launches_of(*d, false, true) + 1;
}

MOE_API moe_status moe_forward_mxfp8(const moe_dims* d, const void* hidden,
                                     const float* router_logits, const void* w_gate_up_q,
                                     const void* w_gate_up_s, const void* w_down_q,
                                     const void* w_down_s, const void* ws_gate_up_q,
                                     const void* ws_gate_up_s, const void* ws_down_q,
                                     const void* ws_down_s, const void* w_g, void* out,
                                     int32_t* topk_ids_out, float* topk_w_out,
                                     int32_t* expert_counts_out, void* workspace,
                                     size_t workspace_bytes, void* cuda_stream) {
    ExpertWeights W{};
    W.mx = true;
    W.gate_up = w_gate_up_q;
    W.down = w_down_q;
    W.s_gate_up = ws_gate_up_q;
    W.s_down = ws_down_q;
    W.gate_up_sc = static_cast<const uint8_t*>(w_gate_up_s);
    W.down_sc = static_cast<const uint8_t*>(w_down_s);
    W.s_gate_up_sc = static_cast<const uint8_t*>(ws_gate_up_s);
    W.s_down_sc = static_cast<const uint8_t*>(ws_down_s);
    return forward_impl(d, hidden, router_logits, nullptr, nullptr, W, w_g, out, topk_ids_out,
                        topk_w_out, expert_counts_out, workspace, workspace_bytes, cuda_stream);
}

MOE_API moe_status moe_forward_nvfp4(
    const moe_dims* d, const void* hidden, const float* router_logits, const void* w_gate_up_q,
    const void* w_gate_up_s, const float* w_gate_up_g, const void* w_down_q, const void* w_down_s,
    const float* w_down_g, const void* ws_gate_up_q, const void* ws_gate_up_s,
    const float* ws_gate_up_g, const void* ws_down_q, const void* ws_down_s, const float* ws_down_g,
    const void* w_g, void* out, int32_t* topk_ids_out, float* topk_w_out,
    int32_t* expert_counts_out, void* workspace, size_t workspace_bytes, void* cuda_stream) {
    ExpertWeights W{};
    W.mx = true;
    W.nv = true;
    W.gate_up = w_gate_up_q;
    W.down = w_down_q;
    W.s_gate_up = ws_gate_up_q;
    W.s_down = ws_down_q;
    W.gate_up_sc = static_cast<const uint8_t*>(w_gate_up_s);
    W.down_sc = static_cast<const uint8_t*>(w_down_s);
    W.s_gate_up_sc = static_cast<const uint8_t*>(ws_gate_up_s);
    W.s_down_sc = static_cast<const uint8_t*>(ws_down_s);
    W.g_gate_up = w_gate_up_g;
    W.g_down = w_down_g;
    W.g_s_gate_up = ws_gate_up_g;
    W.g_s_down = ws_down_g;
    return forward_impl(d, hidden, router_logits, nullptr, nullptr, W, w_g, out, topk_ids_out,
                        topk_w_out, expert_counts_out, workspace, workspace_bytes, cuda_stream);
}

MOE_API moe_status moe_nvfp4_dequant(const void* codes, const void* scales, int rows, int cols,
                                     void* out, void* cuda_stream) {
    if (rows < 0 || cols < 0 || cols % 32 != 0) return MOE_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return MOE_OK;
    if (!codes || !scales || !out || !aligned16(codes) || !aligned16(out))
        return MOE_ERR_INVALID_ARG;
    if (launch_nvfp4_dequant(static_cast<const uint8_t*>(codes),
                             static_cast<const uint8_t*>(scales), rows, cols,
                             static_cast<__nv_bfloat16*>(out),
                             static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

MOE_API moe_status moe_mxfp8_dequant(const void* codes, const void* scales, int rows, int cols,
                                     void* out, void* cuda_stream) {
    if (rows < 0 || cols < 0 || cols % 32 != 0) return MOE_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return MOE_OK;
    if (!codes || !scales || !out || !aligned16(codes) || !aligned16(out))
        return MOE_ERR_INVALID_ARG;
    if (launch_mxfp8_dequant(static_cast<const uint8_t*>(codes),
                             static_cast<const uint8_t*>(scales), rows, cols,
                             static_cast<__nv_bfloat16*>(out),
                             static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

MOE_API int moe_launch_count(const moe_dims* d) {
    if (!dims_valid(d) || !dims_supported(d) || d->T == 0) return 0;
    return launches_of(*d, false);
}

MOE_API int moe_launch_count_quantized(const moe_dims* d) {
    if (!dims_valid(d) || !dims_supported(d) || !dims_supported_mx(d) || d->T == 0) return 0;
    return launches_of(*d, true);
}

MOE_API void moe_set_expert_fusion(int enable) {
    tl_fusion = enable <= 0 ? 0 : (enable >= 2 ? 2 : 1);
}

MOE_API int moe_get_expert_fusion(void) { return tl_fusion; }

MOE_API moe_status moe_set_stage_events(void* const* events, int n_events) {
    if (n_events == 0 || events == nullptr) {
        tl_stage_events_on = false;
        return MOE_OK;
    }
    if (n_events != MOE_NUM_STAGES + 1) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < n_events; ++i) {
        if (!events[i]) return MOE_ERR_INVALID_ARG;
        tl_stage_events[i] = static_cast<cudaEvent_t>(events[i]);
    }
    tl_stage_events_on = true;
    return MOE_OK;
}

namespace moe {
// moe_route.cu: n (a multiple of 32) fp32 values through the y16 format.
cudaError_t launch_y16_roundtrip(long n, const float* in, float* out, cudaStream_t st);
}  // namespace moe

MOE_API moe_status moe_y16_roundtrip(const float* in, float* out, int64_t n, void* cuda_stream) {
    if (n < 0 || n % 32 != 0) return MOE_ERR_INVALID_ARG;
    if (n == 0) return MOE_OK;
    if (!in || !out) return MOE_ERR_INVALID_ARG;
    if (launch_y16_roundtrip(static_cast<long>(n), in, out, static_cast<cudaStream_t>(cuda_stream)) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

MOE_API moe_status moe_selftest_wait_limit(void* workspace, void* cuda_stream) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
        return MOE_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    unsigned* err = static_cast<unsigned*>(workspace);
    if (cudaMemsetAsync(err, 0, sizeof(unsigned), st) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_wait_limit_selftest(err, st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

MOE_API moe_status moe_device_status(const void* workspace, void* cuda_stream) {
    if (!workspace) return MOE_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    unsigned flags = 0;
    if (cudaMemcpy(&flags, workspace, sizeof(flags), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    if (flags & ERR_EP_COUNTS) return MOE_ERR_INVALID_ARG;
    return flags ? MOE_ERR_DEVICE_TIMEOUT : MOE_OK;
}

// ================================================================ expert parallelism
namespace moe {
namespace {

bool ep_dims_valid(const moe_ep_dims* d) {
    if (!d) return false;
    const moe_dims base{d->T, d->H, d->E, d->k, d->I, d->I_s, d->score_fn};
    if (!dims_valid(&base)) return false;
    if (d->G < 1 || d->G > d->E || d->E % d->G != 0) return false;
    if (d->R_max < 0 || d->R_max > (1 << 27)) return false;
    return true;
}

bool ep_dims_supported(const moe_ep_dims* d) {
    const moe_dims base{d->T, d->H, d->E, d->k, d->I, d->I_s, d->score_fn};
    return dims_supported(&base);
}

// Workspace of one rank: the routing arrays of its T tokens (the first part
// of the single-GPU layout, status block first), then the GEMM arrays sized
// for R_max received rows plus the rank's T shared-expert rows.
struct EpLayout {
    size_t meta, blockhist, topk_ids, topk_w, gate_logit, counts, offsets, perm, inv;
    size_t rt_gu, rt_dn, h_hi, h_lo, hs_hi, hs_lo, y, total;
};

EpLayout ep_layout_of(const moe_ep_dims& d) {
    EpLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + (bytes ? bytes : 1), kAlign);
        return o;
    };
    const size_t T = d.T, H = d.H, E = d.E, I = d.I, Is = d.I_s, tk = T * d.k, R = d.R_max;
    const size_t nb = (T + kCountTokens - 1) / kCountTokens;
    L.meta = take(META_WORDS * sizeof(int));
    L.blockhist = take(nb * E * 4);
    L.topk_ids = take(tk * 4);
    L.topk_w = take(tk * 4);
    L.gate_logit = take(T * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.perm = take(tk * 4);
    L.inv = take(tk * 4);
    // row tiles: those the routing writes for the local batch, or those of the
    // received rows (G * E / G segments), whichever list is longer
    const size_t rt = std::max(max_row_tiles(tk, E, 16), max_row_tiles(R, E, 16));
    L.rt_gu = take(rt * sizeof(int4));
    L.rt_dn = take(rt * sizeof(int4));
    L.h_hi = take(R * I * 2);
    L.h_lo = take(R * I * 2);
    L.hs_hi = take(T * Is * 2);
    L.hs_lo = take(T * Is * 2);
    L.y = take((R + T) * H * 4);
    L.total = off;
    return L;
}

bool ep_workspace_ok(const moe_ep_dims& d, const void* workspace, size_t bytes) {
    return workspace && bytes >= ep_layout_of(d).total &&
           (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) == 0;
}

}  // namespace
}  // namespace moe

MOE_API size_t moe_ep_workspace_size(const moe_ep_dims* d) {
    if (!ep_dims_valid(d)) return 0;
    return ep_layout_of(*d).total;
}

MOE_API moe_status moe_ep_workspace_layout(const moe_ep_dims* d, moe_ep_layout_t* out) {
    if (!ep_dims_valid(d) || !out) return MOE_ERR_INVALID_ARG;
    const EpLayout L = ep_layout_of(*d);
    out->topk_ids = L.topk_ids;
    out->topk_w = L.topk_w;
    out->gate_logit = L.gate_logit;
    out->counts = L.counts;
    out->offsets = L.offsets;
    out->perm = L.perm;
    out->inv = L.inv;
    out->y = L.y;
    out->total = L.total;
    return MOE_OK;
}

MOE_API moe_status moe_ep_dispatch(const moe_ep_dims* d, const void* hidden,
                                   const float* router_logits, const void* w_g, void* x_send,
                                   int32_t* send_counts, int32_t* topk_ids_out,
                                   float* topk_w_out, void* workspace, size_t workspace_bytes,
                                   void* cuda_stream) {
    if (!ep_dims_valid(d)) return MOE_ERR_INVALID_ARG;
    if (!ep_dims_supported(d)) return MOE_ERR_UNSUPPORTED;
    if (!send_counts || (reinterpret_cast<uintptr_t>(send_counts) & 3u)) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    if (d->T == 0) {  // nothing routed: every count is zero
        return cudaMemsetAsync(send_counts, 0, sizeof(int32_t) * d->E, st) == cudaSuccess
                   ? MOE_OK
                   : MOE_ERR_CUDA;
    }
    const void* required[] = {hidden, router_logits, w_g, x_send};
    for (const void* p : required)
        if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    const void* optional[] = {topk_ids_out, topk_w_out};
    for (const void* p : optional)
        if (p && (reinterpret_cast<uintptr_t>(p) & 3u)) return MOE_ERR_INVALID_ARG;
    if (!ep_workspace_ok(*d, workspace, workspace_bytes)) return MOE_ERR_WORKSPACE;
    const int T = d->T, H = d->H, E = d->E, k = d->k;
    const EpLayout L = ep_layout_of(*d);
    char* ws = static_cast<char*>(workspace);
    int* meta = reinterpret_cast<int*>(ws + L.meta);
    const RouteBufs rb{reinterpret_cast<int*>(ws + L.topk_ids),
                       reinterpret_cast<float*>(ws + L.topk_w),
                       reinterpret_cast<float*>(ws + L.gate_logit),
                       reinterpret_cast<int*>(ws + L.blockhist),
                       reinterpret_cast<int*>(ws + L.counts),
                       reinterpret_cast<int*>(ws + L.offsets),
                       reinterpret_cast<int*>(ws + L.perm),
                       reinterpret_cast<int*>(ws + L.inv),
                       reinterpret_cast<int4*>(ws + L.rt_gu),
                       reinterpret_cast<int4*>(ws + L.rt_dn),
                       meta};
    Layout base{};
    base.meta = L.meta;
    base.blockhist = L.blockhist;
    if (cudaMemsetAsync(meta, 0, routing_zero_bytes(base, T, E, k), st) != cudaSuccess)
        return MOE_ERR_CUDA;
    // The routing's own row tiles are not used here; any supported width will do.
    const LogitSrc lsrc{router_logits, 1, 0, nullptr};
    if (enqueue_routing(T, H, E, k, d->score_fn, 16, 16, lsrc, false, hidden, w_g, rb,
                        topk_ids_out, topk_w_out, send_counts, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_gather_rows(T * k, H, k, rb.perm, static_cast<const __nv_bfloat16*>(hidden),
                           static_cast<__nv_bfloat16*>(x_send), st) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

MOE_API moe_status moe_ep_experts(const moe_ep_dims* d, int32_t R, const void* x_recv,
                                  const int32_t* recv_counts, const void* hidden,
                                  const void* w_gate_up, const void* w_down,
                                  const void* ws_gate_up, const void* ws_down, void* workspace,
                                  size_t workspace_bytes, void* cuda_stream) {
    if (!ep_dims_valid(d)) return MOE_ERR_INVALID_ARG;
    if (!ep_dims_supported(d)) return MOE_ERR_UNSUPPORTED;
    if (R < 0 || R > d->R_max) return MOE_ERR_INVALID_ARG;
    const void* required[] = {recv_counts, w_gate_up, w_down, ws_gate_up, ws_down};
    for (const void* p : required)
        if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (R > 0 && (!x_recv || !aligned16(x_recv))) return MOE_ERR_INVALID_ARG;
    if (d->T > 0 && (!hidden || !aligned16(hidden))) return MOE_ERR_INVALID_ARG;
    if (!ep_workspace_ok(*d, workspace, workspace_bytes)) return MOE_ERR_WORKSPACE;
    if (R == 0 && d->T == 0) return MOE_OK;
    const int T = d->T, H = d->H, G = d->G, I = d->I, Is = d->I_s;
    const int E_loc = d->E / G;
    const EpLayout L = ep_layout_of(*d);
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    char* ws = static_cast<char*>(workspace);
    int* meta = reinterpret_cast<int*>(ws + L.meta);
    int4* rt_gu = reinterpret_cast<int4*>(ws + L.rt_gu);
    int4* rt_dn = reinterpret_cast<int4*>(ws + L.rt_dn);
    auto* h_hi = reinterpret_cast<__nv_bfloat16*>(ws + L.h_hi);
    auto* hs_hi = reinterpret_cast<__nv_bfloat16*>(ws + L.hs_hi);
    float* y = reinterpret_cast<float*>(ws + L.y);
    const int num_sms = sm_count();
    if (num_sms <= 0) return MOE_ERR_CUDA;

    // Tile widths from the mean rows per (source, local expert) segment; the
    // down GEMM keeps the weights on M (at most 64 tokens per tile) so that y
    // is fp32 on every rank.
    const size_t segs = static_cast<size_t>(G) * E_loc;
    const int bn_gu = pick_bn(static_cast<size_t>(R), static_cast<int>(segs), 256, true);
    const int bn_dn = pick_bn(static_cast<size_t>(R), static_cast<int>(segs), 64, false);

    GemmMaps gu{}, dn{};
    const uint64_t Rm = R > 0 ? R : 1, Tm = T > 0 ? T : 1;  // maps need non-empty dimensions
    const uint32_t gu_rows = static_cast<uint32_t>(gate_up_ts_features(bn_gu));
    bool ok = make_pair_map(&gu.w, w_gate_up, H, static_cast<uint64_t>(E_loc) * 2 * I - I,
                            static_cast<uint64_t>(I) * H * 2, gu_rows) &&
              make_pair_map(&gu.ws, ws_gate_up, H, Is, static_cast<uint64_t>(Is) * H * 2, gu_rows) &&
              make_down_maps(&dn, w_down, ws_down, h_hi, hs_hi, L.h_lo - L.h_hi, L.hs_lo - L.hs_hi,
                             E_loc, H, I, Is, Tm, Rm, bn_dn, false) &&
              make_store_map(&dn.st[0], y, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H,
                             static_cast<uint64_t>(R) + T);
    if (!ok) return MOE_ERR_CUDA;

    GemmArgs ga{};
    ga.T = T;
    ga.H = H;
    ga.E = E_loc;
    ga.k = 1;
    ga.I = I;
    ga.I_s = Is;
    ga.P = R;
    ga.hidden = static_cast<const __nv_bfloat16*>(hidden);
    ga.xrows = static_cast<const __nv_bfloat16*>(x_recv);
    ga.meta = meta;
    ga.gate_logit = reinterpret_cast<const float*>(ws + L.gate_logit);
    ga.h_hi = h_hi;
    ga.h_lo = reinterpret_cast<__nv_bfloat16*>(ws + L.h_lo);
    ga.hs_hi = hs_hi;
    ga.hs_lo = reinterpret_cast<__nv_bfloat16*>(ws + L.hs_lo);
    ga.y = y;
    ga.err = reinterpret_cast<unsigned*>(meta + META_ERR);
    GemmArgs gd = ga;
    ga.rowtiles = rt_gu;
    gd.rowtiles = rt_dn;
    ga.sched = meta + META_SCHED_GU;
    gd.sched = meta + META_SCHED_DN;

    const size_t routed_min = static_cast<size_t>(R) < segs ? static_cast<size_t>(R) : segs;
    const int F_gu = (I + static_cast<int>(gu_rows) - 1) / static_cast<int>(gu_rows);
    const int F_s = (Is + static_cast<int>(gu_rows) - 1) / static_cast<int>(gu_rows);
    const int F_dn = bn_dn == 64 ? (H + 255) / 256 : (H + kGemmBM - 1) / kGemmBM;
    const size_t max_gu = (R / bn_gu + routed_min) * F_gu + ((T + bn_gu - 1) / bn_gu) * F_s;
    const size_t max_dn = (R / bn_dn + routed_min) * F_dn + ((T + bn_dn - 1) / bn_dn) * F_dn;
    const size_t cap = 1u << 30;
    const int tiles_gu = static_cast<int>(max_gu < cap ? max_gu : cap);
    const int tiles_dn = static_cast<int>(max_dn < cap ? max_dn : cap);

    if (cudaMemsetAsync(meta, 0, META_WORDS * sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_ep_tiles(G, E_loc, R, recv_counts, bn_gu, bn_dn, rt_gu, rt_dn, meta, st) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_gate_up(bn_gu, gu, ga, tiles_gu, num_sms, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_down(bn_dn, dn, gd, tiles_dn, num_sms, st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

MOE_API moe_status moe_ep_combine(const moe_ep_dims* d, int32_t R, const float* y_back,
                                  void* out, void* workspace, size_t workspace_bytes,
                                  void* cuda_stream) {
    if (!ep_dims_valid(d)) return MOE_ERR_INVALID_ARG;
    if (!ep_dims_supported(d)) return MOE_ERR_UNSUPPORTED;
    if (R < 0 || R > d->R_max) return MOE_ERR_INVALID_ARG;
    if (d->T == 0) return MOE_OK;
    if (!y_back || !aligned16(y_back) || !out || !aligned16(out)) return MOE_ERR_INVALID_ARG;
    if (!ep_workspace_ok(*d, workspace, workspace_bytes)) return MOE_ERR_WORKSPACE;
    const EpLayout L = ep_layout_of(*d);
    char* ws = static_cast<char*>(workspace);
    const float* y_shared = reinterpret_cast<const float*>(ws + L.y) + static_cast<size_t>(R) * d->H;
    if (launch_combine_split(d->T, d->H, d->k, y_back, y_shared,
                             reinterpret_cast<const float*>(ws + L.topk_w),
                             reinterpret_cast<const int*>(ws + L.inv),
                             static_cast<__nv_bfloat16*>(out),
                             static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
