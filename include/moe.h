/*
 * libmoe: the FFN-side Mixture-of-Experts layer of a Qwen3.5-style hybrid
 * model on one Blackwell (sm_103a) GPU, behind a plain C ABI.
 *
 * The layer sits at the attention-to-experts boundary described in
 * "[RFC] Experimental Qwen3.5 MoE AFD support: CUDA correctness baseline"
 * (Proposed plugin boundary): it receives the hidden states and one fp32
 * router-logit row per token, runs the routed experts and the shared expert,
 * and returns the expert output. The residual add stays with the caller.
 *
 * Per token t with hidden row x (bf16, length H) and logit row l (fp32,
 * length E):
 *   1. score   s_e = softmax_e(l) or sigmoid(l_e)          (selectable)
 *   2. select  the k experts with the largest logits, ties to the lower
 *              expert index, ordered by descending logit
 *   3. weight  w_j = s_{e_j} / sum_j' s_{e_j'}             (top-k renorm)
 *   4. expert  y_j = W_down[e_j] (silu(G x) * (U x)),  G = W_gate_up[e_j][0:I],
 *              U = W_gate_up[e_j][I:2I]                     (SwiGLU)
 *   5. shared  y_s = Ws_down (silu(Gs x) * (Us x)), gated by sigmoid(x . w_g)
 *   6. output  out = bf16( sum_j w_j y_j + sigmoid(x . w_g) y_s )
 * Sources: "Add Qwen3.5-35B-A3B (support vision and text input)":
 * Description (top-8 of 256 experts, per-token sigmoid-gated shared expert,
 * stacked 3D expert weights), Model Information (sigmoid routing) and
 * Additional Information (router in fp32, softmax score, normalize top-k
 * affinities).
 *
 * Conventions for every entry point:
 *   - Tensor arguments are DEVICE pointers to contiguous row-major arrays,
 *     owned by the caller, 16-byte aligned. The library keeps no pointer
 *     after a call returns and allocates no device memory (the one
 *     exception: the host-memory serving loop, moe_pipeline_*, below).
 *   - bf16 arrays are passed as void* (IEEE bfloat16 bit patterns).
 *   - Work is enqueued on the caller's CUDA stream (cudaStream_t passed as
 *     void*; NULL = legacy default stream) without a host synchronisation;
 *     results are valid once the stream has reached that point.
 *   - Calls that share one workspace must not overlap on the GPU.
 */
#ifndef LIBMOE_MOE_H
#define LIBMOE_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_SCORE_SOFTMAX = 0, /* softmax over all E logits of the token */
    MOE_SCORE_SIGMOID = 1  /* independent sigmoid of each logit */
} moe_score_fn;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer */
    MOE_ERR_UNSUPPORTED = 2,   /* H, I or I_s not a multiple of 64 (128: MXFP8, NVFP4) */
    MOE_ERR_WORKSPACE = 3,     /* workspace null or smaller than moe_workspace_size() */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime or driver call failed */
    MOE_ERR_DEVICE_TIMEOUT = 5, /* a kernel gave up waiting on an internal pipeline
                                   barrier and returned early; outputs are invalid */
    MOE_ERR_CAPACITY = 6        /* sizes exceed the fixed scratch of moe_expert_counts_static */
} moe_status;

/* Problem sizes. T tokens, hidden size H, E routed experts, top-k, expert
 * intermediate size I, shared-expert intermediate size I_s, and the score
 * function (a moe_score_fn value).
 * Limits: 0 <= T <= 2^22; 1 <= k <= E <= 1024; k <= 32; H, I, I_s in
 * [64, 65536] and multiples of 64 (else MOE_ERR_UNSUPPORTED). */
typedef struct {
    int32_t T, H, E, k, I, I_s;
    int32_t score_fn;
} moe_dims;

/* Bytes of device workspace moe_forward needs for these sizes (0 if the
 * sizes are invalid). The workspace holds the routing results, the
 * per-expert token lists, the SwiGLU activations and the per-slot expert
 * outputs; its size grows as T * (k + 1) * H * 4 bytes plus lower-order
 * terms. */
size_t moe_workspace_size(const moe_dims* d);

/*
 * Run the layer.
 *   hidden        [T, H]       bf16   normed hidden states
 *   router_logits [T, E]       fp32   router logits (computed upstream)
 *   w_gate_up     [E, 2I, H]   bf16   rows [0, I) gate, rows [I, 2I) up
 *   w_down        [E, H, I]    bf16
 *   ws_gate_up    [2I_s, H]    bf16   shared expert, same row convention
 *   ws_down       [H, I_s]     bf16
 *   w_g           [H]          bf16   shared-expert gate vector
 *   out           [T, H]       bf16   expert output (written)
 *   topk_ids_out  [T, k]       int32  selected experts, in ranking order (NULL: not returned)
 *   topk_w_out    [T, k]       fp32   renormalised weights (NULL: not returned)
 *   expert_counts_out [E]      int32  tokens routed to each expert (NULL: not returned)
 *   workspace     device buffer of at least moe_workspace_size(d) bytes,
 *                 256-byte aligned; its contents need no initialisation
 *   cuda_stream   cudaStream_t as void*
 * Returns MOE_OK after enqueueing every kernel. T = 0 returns MOE_OK and
 * enqueues nothing. Errors detected on the host return before anything is
 * enqueued. Non-finite logits give an unspecified (but in-range) routing.
 * Device-side pipeline timeouts are reported by moe_device_status().
 */
moe_status moe_forward(const moe_dims* d, const void* hidden, const float* router_logits,
                       const void* w_gate_up, const void* w_down, const void* ws_gate_up,
                       const void* ws_down, const void* w_g, void* out, int32_t* topk_ids_out,
                       float* topk_w_out, int32_t* expert_counts_out, void* workspace,
                       size_t workspace_bytes, void* cuda_stream);

/*
 * Serving loop from host memory: moe_forward fed from host buffers, with the
 * output returned into host buffers, and the host<->device copies of
 * neighbouring steps overlapping the compute. The layer, its arithmetic and
 * its results are moe_forward's; this is the host-side runtime around it.
 *
 * moe_pipeline_create(d, w_gate_up, w_down, ws_gate_up, ws_down, w_g,
 *                     cuda_stream, &p)
 *   d and the weight pointers as for moe_forward (device pointers, kept by
 *   the pipeline until it is destroyed: the weights must outlive it); T >= 1.
 *   Unlike every other entry point, this one allocates device memory: two
 *   staging sets of hidden [T, H] bf16, logits [T, E] fp32 and out [T, H]
 *   bf16, one moe_forward workspace, two copy streams (non-blocking) and six
 *   events, all on the current device and freed by moe_pipeline_destroy.
 *   Compute runs on cuda_stream. Returns MOE_ERR_INVALID_ARG (null
 *   pointers, invalid sizes, T = 0) or MOE_ERR_CUDA (an allocation failed;
 *   nothing is left allocated), with *p = NULL on any error.
 * moe_pipeline_submit(p, hidden_host, logits_host, out_host)
 *   One step. hidden_host [T, H] bf16 and logits_host [T, E] fp32 are host
 *   buffers (pinned for the copies to be asynchronous) copied in on the
 *   pipeline's input stream; out_host [T, H] bf16 (host) receives the output
 *   on its output stream. Step i uses staging set i % 2: its input copy waits
 *   only for step i - 2's compute, so it overlaps step i - 1's compute; the
 *   compute waits for its inputs and for step i - 2's output copy; the output
 *   copy waits for the compute. The host buffers of a step must stay
 *   unchanged (inputs) and unread (output) until moe_pipeline_drain returns
 *   or two further steps have been submitted and drained. Returns after
 *   enqueueing (no host synchronisation): MOE_ERR_INVALID_ARG for null
 *   buffers, moe_forward's status otherwise, MOE_ERR_CUDA if a copy or event
 *   call failed.
 * moe_pipeline_drain(p)
 *   Waits for every submitted step; returns moe_device_status of the
 *   workspace (MOE_OK, or MOE_ERR_DEVICE_TIMEOUT), or MOE_ERR_CUDA.
 * moe_pipeline_streams(p, &in_stream, &out_stream)
 *   The pipeline's copy streams (cudaStream_t as void*; either output may be
 *   NULL), e.g. to record timing events after the last output copy.
 * moe_pipeline_destroy(p)
 *   Waits for the pipeline's work and frees everything it allocated; NULL is
 *   a no-op.
 */
typedef struct moe_pipeline moe_pipeline;
moe_status moe_pipeline_create(const moe_dims* d, const void* w_gate_up, const void* w_down,
                               const void* ws_gate_up, const void* ws_down, const void* w_g,
                               void* cuda_stream, moe_pipeline** out);
moe_status moe_pipeline_submit(moe_pipeline* p, const void* hidden_host, const float* logits_host,
                               void* out_host);
moe_status moe_pipeline_drain(moe_pipeline* p);
moe_status moe_pipeline_streams(const moe_pipeline* p, void** in_stream, void** out_stream);
void moe_pipeline_destroy(moe_pipeline* p);

/*
 * Run the layer with MXFP8 expert weights: the same computation as
 * moe_forward, with every weight of the routed and the shared experts given
 * in the OCP Microscaling MXFP8 format instead of bf16. The pages deploy
 * block-FP8 expert banks ("qwen3_5_moe is TP=1-only ...", first comment)
 * without fixing the block format; MXFP8 is the block-scaled FP8 with
 * power-of-two scales:
 *   a weight matrix [rows, K] is stored as
 *     codes  [rows, K]     uint8  FP8 E4M3 (sign, 4-bit exponent with bias 7,
 *                                 3-bit mantissa; exponent 0 = subnormal)
 *     scales [K/32, rows]  uint8  UE8M0: scale code s stands for 2^(s - 127)
 *   and element (r, c) is E4M3(codes[r][c]) * 2^(scales[c/32][r] - 127).
 *   w_gate_up_q [E, 2I, H] codes, w_gate_up_s [E, H/32, 2I] scales
 *   w_down_q    [E, H, I]  codes, w_down_s    [E, I/32, H]  scales
 *   ws_gate_up_q [2I_s, H], ws_gate_up_s [H/32, 2I_s]   (shared expert)
 *   ws_down_q    [H, I_s],  ws_down_s    [I_s/32, H]
 * Each such value has at most 4 significant bits and is exactly a bf16
 * number for scale codes 3..246, so the layer equals moe_forward run on the
 * dequantised bf16 weights (the E4M3 NaN codes and the scale code 255 are
 * reserved: the results are then unspecified). The activations (hidden, h),
 * the router logits and w_g stay as in moe_forward.
 * Sizes: H, I and I_s must be multiples of 128 (else MOE_ERR_UNSUPPORTED).
 * The workspace is the one of moe_workspace_size(d); the h_hi / h_lo
 * regions of moe_workspace_layout then hold h in 64-column panels (panel c:
 * columns 64c..64c+63 of every h_hi row, then of every h_lo row) and y is
 * always fp32. Other arguments, the returns and the error behaviour are
 * those of moe_forward; the scale pointers must be 16-byte aligned.
 */
moe_status moe_forward_mxfp8(const moe_dims* d, const void* hidden, const float* router_logits,
                             const void* w_gate_up_q, const void* w_gate_up_s,
                             const void* w_down_q, const void* w_down_s,
                             const void* ws_gate_up_q, const void* ws_gate_up_s,
                             const void* ws_down_q, const void* ws_down_s, const void* w_g,
                             void* out, int32_t* topk_ids_out, float* topk_w_out,
                             int32_t* expert_counts_out, void* workspace, size_t workspace_bytes,
                             void* cuda_stream);

/*
 * Run the layer with NVFP4 expert weights: the same computation as
 * moe_forward, with every weight matrix of the routed and the shared experts
 * given in NVIDIA's NVFP4 format (the pages deploy NVFP4 expert banks:
 * "qwen3_5_moe is TP=1-only ...", second comment, without fixing a layout):
 *   a weight matrix [rows, K] is stored as
 *     codes  [rows, K/2]   uint8  two FP4 E2M1 values per byte (sign, 2-bit
 *                                 exponent with bias 1, 1-bit mantissa), the
 *                                 lower K index in the low nibble
 *     scales [K/16, rows]  uint8  FP8 E4M3 block scale of each 16 values
 *     g                    fp32   one scale for the whole matrix
 *   and element (r, c) is g * E2M1(value c of row r) * E4M3(scales[c/16][r]).
 *   w_gate_up_q [E, 2I, H/2], w_gate_up_s [E, H/16, 2I], w_gate_up_g [E]
 *   w_down_q    [E, H, I/2],  w_down_s    [E, I/16, H],  w_down_g    [E]
 *   ws_gate_up_q [2I_s, H/2], ws_gate_up_s [H/16, 2I_s], ws_gate_up_g [1]
 *   ws_down_q    [H, I_s/2],  ws_down_s    [I_s/16, H],  ws_down_g    [1]
 * E2M1 x E4M3 is exactly a bf16 number, so the GEMMs run bf16 MMAs on exact
 * values and multiply each matrix's fp32 accumulators by its g (the gate and
 * up projections before SiLU, the down projection before the shared gate and
 * the combine). The E4M3 NaN scale codes are reserved (results unspecified).
 * Sizes: H, I and I_s multiples of 128 (else MOE_ERR_UNSUPPORTED); the g
 * pointers 4-byte aligned, the codes and scales 16-byte aligned. Workspace,
 * other arguments, returns and errors as moe_forward_mxfp8.
 */
moe_status moe_forward_nvfp4(const moe_dims* d, const void* hidden, const float* router_logits,
                             const void* w_gate_up_q, const void* w_gate_up_s,
                             const float* w_gate_up_g, const void* w_down_q, const void* w_down_s,
                             const float* w_down_g, const void* ws_gate_up_q,
                             const void* ws_gate_up_s, const float* ws_gate_up_g,
                             const void* ws_down_q, const void* ws_down_s, const float* ws_down_g,
                             const void* w_g, void* out, int32_t* topk_ids_out, float* topk_w_out,
                             int32_t* expert_counts_out, void* workspace, size_t workspace_bytes,
                             void* cuda_stream);

/* bf16 values E2M1 x E4M3 (without the matrix scale g) of one NVFP4 matrix
 * (layout as in moe_forward_nvfp4): codes [rows, cols/2], scales [cols/16,
 * rows] in, out [rows, cols] bf16 written, with the conversion the NVFP4
 * GEMMs use (exact). cols must be a multiple of 32 (else MOE_ERR_INVALID_ARG);
 * codes and out 16-byte aligned. Enqueued on cuda_stream. */
moe_status moe_nvfp4_dequant(const void* codes, const void* scales, int rows, int cols, void* out,
                             void* cuda_stream);

/* bf16 values of one MXFP8 matrix (layout as in moe_forward_mxfp8): codes
 * [rows, cols] and scales [cols/32, rows] in, out [rows, cols] bf16 written,
 * with the conversion the MXFP8 GEMMs use (exact for scale codes 3..246).
 * cols must be a multiple of 32 (else MOE_ERR_INVALID_ARG); codes and out
 * 16-byte aligned. Enqueued on cuda_stream. */
moe_status moe_mxfp8_dequant(const void* codes, const void* scales, int rows, int cols, void* out,
                             void* cuda_stream);

/*
 * Run the layer with the router on the FFN side: the same computation as
 * moe_forward, with the router logits computed first from the router weights
 * instead of being passed in (the step just before the layer's boundary in
 * "[RFC] Experimental Qwen3.5 MoE AFD support: CUDA correctness baseline",
 * for callers that keep the router with the experts):
 *   w_router   [E, H]  bf16  router weights, one row per expert
 *   logits[t][e] = sum_h hidden[t][h] * w_router[e][h], accumulated in fp32
 *   (the router runs in fp32: "Add Qwen3.5-35B-A3B (support vision and text
 *   input)", Additional Information; the products of bf16 values are exact),
 *   in an order fixed by the sizes and the GPU's SM count (repeat calls on
 *   one GPU give the same bits): a tensor-core GEMM whose K dimension may be
 *   split across CTAs, the routing kernel adding the split partial sums in a
 *   fixed order; the routing then ranks these fp32 logits.
 *   logits_out [T, E] fp32 receives the logits (NULL: not returned).
 * The workspace must hold moe_workspace_size_router(d) bytes. With
 * moe_set_stage_events, stage 0 spans the router GEMM and the routing. Other
 * arguments, returns and errors as moe_forward.
 */
moe_status moe_forward_router(const moe_dims* d, const void* hidden, const void* w_router,
                              const void* w_gate_up, const void* w_down, const void* ws_gate_up,
                              const void* ws_down, const void* w_g, void* out, float* logits_out,
                              int32_t* topk_ids_out, float* topk_w_out,
                              int32_t* expert_counts_out, void* workspace,
                              size_t workspace_bytes, void* cuda_stream);

/* Workspace bytes of moe_forward_router: moe_workspace_size(d) plus the
 * router GEMM's split-K partial sums (0 for invalid sizes). */
size_t moe_workspace_size_router(const moe_dims* d);

/* Kernels one moe_forward_router launches: those of moe_forward plus the
 * router GEMM (0 for invalid sizes or T = 0). */
int moe_launch_count_router(const moe_dims* d);

/* Synchronise cuda_stream, then report MOE_ERR_DEVICE_TIMEOUT if the last
 * moe_forward that used this workspace hit a pipeline timeout, MOE_ERR_CUDA
 * on a CUDA error, else MOE_OK. */
moe_status moe_device_status(const void* workspace, void* cuda_stream);

/* Static, human-readable name of a status code. */
const char* moe_status_string(moe_status s);

/* Byte offsets of the intermediate arrays inside the workspace, for
 * inspection after a call (all arrays row-major):
 *   topk_ids  [T, k] int32, topk_w [T, k] fp32, gate_logit [T] fp32 (x . w_g),
 *   counts [E] int32, offsets [E + 1] int32 (exclusive prefix of counts),
 *   perm [T k] int32 (slot t*k+j at its position in expert-sorted order,
 *   tokens ascending within an expert), inv [T k] int32 (position of slot
 *   t*k+j), h_hi / h_lo [T k, I] bf16 (SwiGLU activation of each routed slot
 *   in sorted order, as a high + low bf16 pair), hs_hi / hs_lo [T, I_s] bf16
 *   (shared expert activation), y [T k + T, H] (rows [0, T k): routed
 *   expert outputs in sorted order; rows T k + t: gated shared output).
 *   y holds fp32 values, except when fp32 y ((T k + T) H 4 bytes) would
 *   exceed 64 MiB or, with bf16 expert weights, when the mean expert group
 *   is large enough for 128-token down tiles (1.25 T k / E > 64): then it
 *   holds y16 codes,
 *   16 bits per value (rows of 2 H bytes) followed by an exponent plane of
 *   one byte per 32 values of each row (row stride H/32 rounded up to a
 *   multiple of 4): a value v of a block with exponent byte b is |v| +
 *   2^(b-127) rounded to a 12-bit significand, stored as 4 exponent bits
 *   relative to b, 11 fraction bits and the sign. The region is sized for
 *   fp32 either way. */
typedef struct {
    size_t topk_ids, topk_w, gate_logit, counts, offsets, perm, inv;
    size_t h_hi, h_lo, hs_hi, hs_lo, y;
    size_t total;
} moe_workspace_layout_t;

moe_status moe_workspace_layout(const moe_dims* d, moe_workspace_layout_t* layout);

/* Stages of one moe_forward, each at most one kernel: routing (with the
 * per-expert histograms and their scan when T*k > 2048; the whole permute
 * when T*k <= 2048), scatter, gate_up GEMM, down GEMM, combine. A stage that
 * a batch merges into the one before is empty: the scatter stage when
 * T*k <= 2048, and the down stage when the fused expert launch
 * (moe_set_expert_fusion, when enabled) runs in the gate_up stage. The
 * whole-layer launch (fusion level 2) runs in the routing stage and leaves the
 * other four empty. */
#define MOE_NUM_STAGES 5

/* Optional per-kernel timing. `events` points to MOE_NUM_STAGES + 1
 * cudaEvent_t handles (passed as void*) created by the caller; while set,
 * every moe_forward issued from the calling host thread records events[i]
 * on its stream just before kernel i and events[MOE_NUM_STAGES] after the
 * last one, so kernel i runs between events[i] and events[i + 1]. Pass NULL
 * (n_events = 0) to stop. The library does not own the events. Returns
 * MOE_ERR_INVALID_ARG unless n_events is 0 or MOE_NUM_STAGES + 1. */
moe_status moe_set_stage_events(void* const* events, int n_events);

/* Number of kernels one moe_forward with these sizes launches from the
 * calling host thread, or 0 for invalid sizes or T = 0: routing (1 launch
 * when T*k <= 2048, else 2), the expert GEMMs (1 launch when they run fused,
 * else 2) and the combine; 1 when the whole layer runs as one launch. */
int moe_launch_count(const moe_dims* d);

/* The same for moe_forward_mxfp8 and moe_forward_nvfp4 (their expert GEMMs
 * always take two launches); 0 also for sizes those entry points reject. */
int moe_launch_count_quantized(const moe_dims* d);

/* Fused expert phase (bf16 weights: moe_forward and moe_forward_router).
 * When enabled (per host thread; off by default) and the batch's gate_up and
 * down token tiles have the same width of at most 64 tokens (decode-sized
 * batches: about T*k/E <= 51 tokens per expert), the two grouped GEMMs run
 * as one persistent launch. Its tile sequence holds the gate_up tiles and
 * then the down tiles; a down tile waits on a device counter (bounded in
 * time, like every wait in the library) for the gate_up tiles of its row
 * tile. That removes the idle tail of the gate_up launch and the refill of
 * the down pipeline. The arithmetic is the same as the two launches', so the
 * results are bitwise identical. Measured on GB300 it is no faster than
 * the two launches at decode and about 4 % slower on wide batches, hence
 * off by default. The wait needs every CTA of the launch
 * resident at once (one per SM); if another kernel holds SMs for longer
 * than the wait limit, the layer reports MOE_ERR_DEVICE_TIMEOUT through
 * moe_device_status. Source: "Add Qwen3.5-35B-A3B (support vision and text
 * input)", Description (the routed experts and the shared expert); the
 * fusion is an implementation choice.
 *
 * enable: 0 (default) separate launches; 1 the fused expert phase above;
 * 2 also, where it applies, the whole layer in one persistent launch of one
 * CTA per SM: moe_forward (router logits given, not moe_forward_router),
 * T*k <= 2048, E <= 256 and the fused expert phase applying (decode-sized
 * batches). In that launch every CTA routes tokens (CTA b takes tokens b,
 * b + #SMs, ...), the last CTA to finish builds the permute, the others wait
 * for it; then the fused expert phase; then every CTA waits until all have
 * finished their expert tiles and combines its tokens. Both waits are bounded
 * in time like every wait in the library (a timeout is reported by
 * moe_device_status as MOE_ERR_DEVICE_TIMEOUT, and no token is combined
 * after one). The arithmetic is that of the separate kernels: results,
 * routing outputs and counts are bitwise identical. Other values are
 * clamped to 0..2. moe_get_expert_fusion returns the calling thread's level. */
void moe_set_expert_fusion(int enable);
int moe_get_expert_fusion(void);

/* Self-test of the kernels' bounded waits (failure detection without a GPU
 * fault): clears the status word at the start of `workspace` (256-byte
 * aligned device memory, at least 4 bytes) and enqueues one CTA on
 * `cuda_stream` that waits on a barrier nothing ever completes, with the same
 * bounded wait the GEMM pipelines use. The wait gives up after its time limit
 * (2 s) and sets a bit of the status word; moe_device_status(workspace,
 * stream) then returns MOE_ERR_DEVICE_TIMEOUT and the context stays usable.
 * Returns MOE_ERR_WORKSPACE for a missing or misaligned workspace. */
moe_status moe_selftest_wait_limit(void* workspace, void* cuda_stream);

/* Test hook of the y16 format in which the down GEMMs hand large expert
 * outputs to the combine (see the workspace layout above): out[i] = the
 * value in[i] decodes to after encoding, each block of 32 consecutive values
 * taking one exponent byte from its largest magnitude. n (a multiple of 32,
 * else MOE_ERR_INVALID_ARG) device fp32 values; enqueued on cuda_stream. */
moe_status moe_y16_roundtrip(const float* in, float* out, int64_t n, void* cuda_stream);

/*
 * Expert parallelism: the layer spread over G ranks (one GPU each), rank g
 * owning the contiguous block of routed experts [g E/G, (g+1) E/G) and a copy
 * of the shared expert; every rank brings its own tokens. The pages run the
 * experts this way ("FastAFD" pull request, What the model needed: expert
 * workers at EP 4; "qwen3_5_moe is TP=1-only ...", first comment: routed
 * experts sharded across ranks). Per rank, with the two exchanges done by the
 * caller (e.g. an NCCL all-to-all) between the calls:
 *   1. moe_ep_dispatch: routing and the permute of the rank's tokens over all
 *      E experts (as in moe_forward), then the hidden rows of its (token,
 *      slot) pairs in expert-sorted order into x_send, and the number of rows
 *      per expert into send_counts. The rows bound for rank g are the
 *      contiguous range of x_send that holds experts [g E/G, (g+1) E/G).
 *   2. exchange: rank g receives, from every source rank s in rank order,
 *      that range of s's x_send and s's counts of g's experts: x_recv [R, H]
 *      (R rows in total) and recv_counts [G, E/G] (row s: source s).
 *   3. moe_ep_experts: the rank's routed experts on the received rows (the
 *      grouped gate_up and down GEMMs of moe_forward) and the shared expert,
 *      gated by sigmoid(x . w_g), on the rank's own tokens. Results in the
 *      workspace (moe_ep_workspace_layout: y): rows [0, R) the expert output
 *      of the received rows, in x_recv's order; rows [R, R + T) the rank's
 *      gated shared-expert rows. All fp32 [., H].
 *   4. exchange back: rows [0, R) of y return to their source ranks (the
 *      reverse of step 2), landing in y_back [T k, H] fp32 in the order of
 *      the rank's own x_send.
 *   5. moe_ep_combine: out = bf16(sum_j w_j y_back[slot j] + shared row),
 *      summed in fp32 in slot order, as in moe_forward (gather, no atomics).
 * moe_forward's results on the same tokens follow from the same arithmetic,
 * except that y is always fp32 here (no y16 codes) and the tile widths depend
 * on the received rows, so outputs agree with moe_forward within the parity
 * tolerance rather than bit for bit.
 */
typedef struct {
    int32_t T;        /* this rank's tokens (0 <= T <= 2^22) */
    int32_t H, E, k, I, I_s, score_fn;  /* as moe_dims; E counts all ranks' experts */
    int32_t G;        /* ranks: 1 <= G <= E, E a multiple of G */
    int32_t R_max;    /* most rows this rank may receive (0 .. 2^27); sizes the workspace */
} moe_ep_dims;

/* Byte offsets inside an expert-parallel workspace (see moe_workspace_layout
 * for the routing arrays): y [R_max + T, H] fp32 holds the expert rows of the
 * last moe_ep_experts call (rows [0, R): received rows, rows [R, R + T): the
 * gated shared-expert rows of the rank's tokens). */
typedef struct {
    size_t topk_ids, topk_w, gate_logit, counts, offsets, perm, inv, y;
    size_t total;
} moe_ep_layout_t;

/* Workspace bytes of one rank (0 for invalid sizes); 256-byte aligned device
 * memory, no initialisation needed. One workspace serves the three calls of a
 * step and must not be shared with concurrent calls. */
size_t moe_ep_workspace_size(const moe_ep_dims* d);
moe_status moe_ep_workspace_layout(const moe_ep_dims* d, moe_ep_layout_t* layout);

/* Step 1. hidden [T, H] bf16, router_logits [T, E] fp32, w_g [H] bf16 as in
 * moe_forward; x_send [T k, H] bf16 and send_counts [E] int32 written;
 * topk_ids_out / topk_w_out [T, k] optional (NULL). T = 0 writes zero counts.
 * Returns MOE_ERR_INVALID_ARG / UNSUPPORTED / WORKSPACE as moe_forward. */
moe_status moe_ep_dispatch(const moe_ep_dims* d, const void* hidden, const float* router_logits,
                           const void* w_g, void* x_send, int32_t* send_counts,
                           int32_t* topk_ids_out, float* topk_w_out, void* workspace,
                           size_t workspace_bytes, void* cuda_stream);

/* Step 3. R received rows (0 <= R <= R_max, else MOE_ERR_INVALID_ARG);
 * x_recv [R, H] bf16 (may be NULL when R = 0); recv_counts [G, E/G] int32 in
 * device memory; hidden [T, H] bf16: the rank's own tokens (the same array
 * given to moe_ep_dispatch, whose gate logits the workspace keeps); the
 * rank's expert weights w_gate_up [E/G, 2I, H], w_down [E/G, H, I] bf16 and
 * the shared expert's ws_gate_up [2I_s, H], ws_down [H, I_s]. Counts that are
 * negative or do not add up to R are detected on the device: no received row
 * is processed and moe_device_status() returns MOE_ERR_INVALID_ARG. */
moe_status moe_ep_experts(const moe_ep_dims* d, int32_t R, const void* x_recv,
                          const int32_t* recv_counts, const void* hidden, const void* w_gate_up,
                          const void* w_down, const void* ws_gate_up, const void* ws_down,
                          void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Step 5. R as given to moe_ep_experts; y_back [T k, H] fp32 (the returned
 * rows, in x_send's order); out [T, H] bf16 written. */
moe_status moe_ep_combine(const moe_ep_dims* d, int32_t R, const float* y_back, void* out,
                          void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * Allocation-free expert histogram. The pages have no counterpart to this
 * entry point; it exists for callers that cannot allocate device memory,
 * for example a plugin behind a fixed interface that receives only its
 * inputs and outputs and has nowhere to keep a workspace, or a
 * latency-critical caller whose device memory is fully pre-reserved and
 * which must not call cudaMalloc (an allocation can synchronise the device).
 *
 * Computes, from a table of selected experts topk_ids [T, k] (int32, device),
 * counts_out [E] (tokens per expert; ids outside [0, E) are not counted) and,
 * if offsets_out is not NULL, offsets_out [E + 1] (exclusive prefix sum of
 * the counts). Same values as moe_forward's expert_counts_out and its
 * workspace offsets for the same routing.
 *
 * Scratch lives in a fixed device array inside the library of
 * MOE_STATIC_HIST_WORDS int32 words (1 MiB) plus a 256-byte header; every
 * GPU that loads the library holds it until the process exits. Sizes with
 * ceil(T / 256) * E > MOE_STATIC_HIST_WORDS return MOE_ERR_CAPACITY (for
 * E = 256: T <= 262144). Limits as for moe_forward otherwise: 1 <= k <= 32,
 * k <= E <= 1024 (else MOE_ERR_INVALID_ARG), so T * k stays below 2^27. The
 * call allocates no memory and calls no allocating library routine. Every
 * call looks up the array's device address in the current device's context
 * (so the address stays valid after a cudaDeviceReset); the first call on a
 * device may also load the library's device code there, so make it before
 * any stream capture. All calls share the array: calls that overlap on the
 * GPU race and give wrong counts. Enqueued on cuda_stream without a host
 * synchronisation.
 */
#define MOE_STATIC_HIST_WORDS (1 << 18)
moe_status moe_expert_counts_static(const int32_t* topk_ids, int32_t T, int32_t k, int32_t E,
                                    int32_t* counts_out, int32_t* offsets_out, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* LIBMOE_MOE_H */
