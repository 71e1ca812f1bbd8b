/*
 * Plain, slow CPU oracle for the FFN-side Mixture-of-Experts layer.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. The CUDA path shares
 * no code with it.
 *
 * Everything is computed in fp64 from the exact values of the bf16 / fp32
 * inputs, with no blocking, fusion or reordering: token by token, expert by
 * expert, dot product by dot product.
 *
 * What the layer computes, and where the pages state it:
 *   - inputs are the hidden states and one fp32 router-logit row per token,
 *     produced on the attention side ("[RFC] Experimental Qwen3.5 MoE AFD
 *     support: CUDA correctness baseline", Proposed plugin boundary; router in
 *     fp32: "Add Qwen3.5-35B-A3B (support vision and text input)", Additional
 *     Information);
 *   - score = softmax over all experts (Additional Information:
 *     router.act_fn=softmax) or per-expert sigmoid (Model Information:
 *     "top-8 sigmoid routing"); selectable;
 *   - top-k selection (Description: top-8 routing over 256 experts), ties to
 *     the lower expert index, order = descending logit;
 *   - renormalise the selected scores to sum to one (Additional Information:
 *     normalize_top_k_affinities=True);
 *   - each selected expert is a SwiGLU FFN on stacked 3D weights
 *     W_gate_up[E, 2I, H] (rows [0, I) gate, [I, 2I) up) and W_down[E, H, I]
 *     (Description: HF stacked 3D expert weights);
 *   - one shared expert, always active, scaled per token by
 *     sigmoid(x . w_g) (Description and Additional Information: per-token
 *     sigmoid-gated shared expert);
 *   - output = sum_j w_j y_j + gate * y_shared, returned as the expert output
 *     (Proposed plugin boundary); no residual add inside the layer.
 *
 * Parity pins (tests/test_oracle_pins.py): brute-force rank selection, tie
 * rows, sum-to-one, closed-form softmax renormalisation, k = E, E = k = 1
 * against a dense SwiGLU evaluated with a library matmul, dense all-expert
 * evaluation with a mask, gate special cases, linearity, token and expert
 * relabelling symmetries. No page prints a worked numeric example of the
 * layer, so exact output values beyond these pins are not fixed by the pages.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_SOFTMAX 0
#define ORACLE_SIGMOID 1

/* Exact value of a bf16 bit pattern. */
static double bf16_value(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Ranking order of the selection: a larger logit ranks first; equal logits
 * rank by the lower expert index. Returns 1 if (va, ia) ranks before (vb, ib). */
static int ranks_before(float va, int ia, float vb, int ib) {
    if (va > vb) return 1;
    if (va < vb) return 0;
    return ia < ib;
}

/*
 * Routing of one token: scores, top-k, renormalisation.
 *   logits  [E] fp32
 *   ids     [k] out, in ranking order
 *   weights [k] out, renormalised selected scores
 * Returns 0, or -1 if the fp64 scores contradict the logit order (which
 * would mean the selection on logits differs from a selection on scores).
 */
int oracle_route_token(int E, int k, int score_fn, const float* logits, int32_t* ids,
                       double* weights) {
    double* score = (double*)malloc(sizeof(double) * (size_t)E);
    char* taken = (char*)calloc((size_t)E, 1);
    if (!score || !taken) { free(score); free(taken); return -2; }

    /* 1. scores, in fp64 from the fp32 logits */
    if (score_fn == ORACLE_SOFTMAX) {
        double m = (double)logits[0];
        for (int e = 1; e < E; ++e)
            if ((double)logits[e] > m) m = (double)logits[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) {
            score[e] = exp((double)logits[e] - m);
            z += score[e];
        }
        for (int e = 0; e < E; ++e) score[e] /= z;
    } else {
        for (int e = 0; e < E; ++e) score[e] = 1.0 / (1.0 + exp(-(double)logits[e]));
    }

    /* 2. selection: k rounds, each takes the best expert not yet taken */
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (taken[e]) continue;
            if (best < 0 || ranks_before(logits[e], e, logits[best], best)) best = e;
        }
        taken[best] = 1;
        ids[j] = best;
    }
    int status = 0;
    for (int j = 1; j < k; ++j)
        if (score[ids[j]] > score[ids[j - 1]]) status = -1;

    /* 3. renormalise the selected scores */
    double sum = 0.0;
    for (int j = 0; j < k; ++j) sum += score[ids[j]];
    for (int j = 0; j < k; ++j) weights[j] = score[ids[j]] / sum;

    free(score);
    free(taken);
    return status;
}

/* Routing of all T tokens. ids [T,k], weights [T,k]. Returns the number of
 * tokens whose score order disagreed with the logit order (0 expected). */
int oracle_route(int T, int E, int k, int score_fn, const float* logits, int32_t* ids,
                 double* weights) {
    int bad = 0;
    for (int t = 0; t < T; ++t)
        if (oracle_route_token(E, k, score_fn, logits + (size_t)t * E, ids + (size_t)t * k,
                               weights + (size_t)t * k) != 0)
            ++bad;
    return bad;
}

/* Tokens routed to each expert. counts [E]. */
void oracle_expert_counts(int T, int E, int k, const int32_t* ids, int32_t* counts) {
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) counts[ids[(size_t)t * k + j]] += 1;
}

/*
 * MXFP8 expert weights (OCP Microscaling formats, MXFP8 with E4M3 elements):
 * each run of 32 consecutive K elements of a weight row shares one UE8M0
 * scale 2^(s - 127); an element is an FP8 E4M3 code (sign, 4-bit exponent
 * with bias 7, 3-bit mantissa; exponent 0 holds the subnormals m * 2^-9;
 * S.1111.111 is NaN; there are no infinities). The pages name block-FP8
 * expert banks ("qwen3_5_moe is TP=1-only ...", first comment) without a
 * block layout; this is the plainest block-scaled FP8 with power-of-two
 * scales.
 */
static double e4m3_value(uint8_t b) {
    const int sign = b >> 7, e = (b >> 3) & 0xF, m = b & 7;
    double v;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

static double ue8m0_value(uint8_t s) { return s == 255 ? NAN : ldexp(1.0, (int)s - 127); }

/* bf16 bit pattern of a double that bf16 represents exactly (finite, at most
 * 8 significant bits, normal or subnormal range); returns -1 if it does not. */
static int32_t exact_bf16_bits(double v) {
    float f = (float)v;
    if ((double)f != v) return -1;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (u & 0xFFFFu) return -1;
    return (int32_t)(u >> 16);
}

/*
 * Dequantise an MXFP8 matrix of `rows` rows and `cols` K elements (cols a
 * multiple of 32): codes [rows, cols], scales [cols / 32, rows] (the scale of
 * row r, K block j at j * rows + r). Every value is exactly a bf16 value
 * (at most 4 significant bits); out gets its bf16 bit pattern. Returns the
 * number of elements that were not exact (NaN codes or scales, or results
 * outside the bf16 range).
 */
int oracle_mxfp8_to_bf16(int rows, int cols, const uint8_t* codes, const uint8_t* scales,
                         uint16_t* out) {
    int bad = 0;
    for (int r = 0; r < rows; ++r)
        for (int c = 0; c < cols; ++c) {
            const double v = e4m3_value(codes[(size_t)r * cols + c]) *
                             ue8m0_value(scales[(size_t)(c / 32) * rows + r]);
            const int32_t bits = exact_bf16_bits(v);
            if (bits < 0) {
                ++bad;
                out[(size_t)r * cols + c] = 0x7FC0u;
            } else {
                out[(size_t)r * cols + c] = (uint16_t)bits;
            }
        }
    return bad;
}

/* Value table of the 256 E4M3 codes (for the oracle's pins). */
void oracle_e4m3_table(double* out) {
    for (int b = 0; b < 256; ++b) out[b] = e4m3_value((uint8_t)b);
}

/*
 * NVFP4 expert weights (the pages deploy NVFP4 expert banks: "qwen3_5_moe is
 * TP=1-only ...", second comment; the format is NVIDIA's NVFP4): FP4 E2M1
 * elements (sign, 2-bit exponent with bias 1, 1-bit mantissa; exponent 0
 * holds 0 and 0.5), two per byte with the lower K index in the low nibble;
 * one FP8 E4M3 scale per 16 consecutive K values of a row; one fp32 scale
 * per weight matrix, applied by the layer to that matrix's products.
 */
static double e2m1_value(uint8_t nib) {
    const int sign = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
    const double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

/* Value table of the 16 E2M1 codes (for the oracle's pins). */
void oracle_e2m1_table(double* out) {
    for (int b = 0; b < 16; ++b) out[b] = e2m1_value((uint8_t)b);
}

/*
 * Dequantise an NVFP4 matrix of `rows` rows and `cols` K values (cols a
 * multiple of 16) without its fp32 matrix scale: codes [rows, cols / 2]
 * (value c of row r in byte c / 2, low nibble for even c), scales
 * [cols / 16, rows] E4M3 (row r, block j at j * rows + r). Every E2M1 x E4M3
 * product has at most 6 significant bits and lies within [2^-10, 2688], so it
 * is exactly a bf16 value; out gets its bit pattern. Returns the number of
 * elements that were not exact (NaN scales).
 */
int oracle_nvfp4_to_bf16(int rows, int cols, const uint8_t* codes, const uint8_t* scales,
                         uint16_t* out) {
    int bad = 0;
    for (int r = 0; r < rows; ++r)
        for (int c = 0; c < cols; ++c) {
            const uint8_t byte = codes[(size_t)r * (cols / 2) + c / 2];
            const uint8_t nib = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
            const double v = e2m1_value(nib) * e4m3_value(scales[(size_t)(c / 16) * rows + r]);
            const int32_t bits = exact_bf16_bits(v);
            if (bits < 0) {
                ++bad;
                out[(size_t)r * cols + c] = 0x7FC0u;
            } else {
                out[(size_t)r * cols + c] = (uint16_t)bits;
            }
        }
    return bad;
}

/*
 * Router logits computed on the FFN side: l[t][e] = sum over h of
 * x[t][h] * W_router[e][h], with W_router [E, H] bf16 (one row per expert,
 * the layout of a linear layer's weight). The router runs in fp32 ("Add
 * Qwen3.5-35B-A3B (support vision and text input)", Additional Information:
 * router dtype float32): every product of two bf16 values is exact, the
 * oracle sums them in fp64 in the natural order of h; out [T, E] holds the
 * fp64 sums (the routing ranks them after one rounding to fp32).
 */
void oracle_router_logits(int T, int H, int E, const uint16_t* hidden, const uint16_t* w_router,
                          double* out) {
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += bf16_value(hidden[(size_t)t * H + h]) *
                       bf16_value(w_router[(size_t)e * H + h]);
            out[(size_t)t * E + e] = acc;
        }
}

static double silu(double g) { return g / (1.0 + exp(-g)); }

/*
 * One SwiGLU FFN applied to one token, with the weight matrices s_gu * W_gu
 * and s_d * W_d (s = 1 for bf16 weights; the fp32 matrix scale of NVFP4
 * weights otherwise, multiplied into each dot product of the matrix):
 *   g_i = s_gu (W_gu[i, :] . x),  u_i = s_gu (W_gu[I + i, :] . x)   (i < I)
 *   a_i = silu(g_i) * u_i
 *   y_h = s_d (W_d[h, :] . a)                                      (h < H)
 * w_gu [2I, H] and w_d [H, I] are bf16 bit patterns; x is fp64 [H].
 */
static void swiglu_ffn(int H, int I, const uint16_t* w_gu, const uint16_t* w_d, double s_gu,
                       double s_d, const double* x, double* a_scratch, double* y) {
    for (int i = 0; i < I; ++i) {
        const uint16_t* wg = w_gu + (size_t)i * H;
        const uint16_t* wu = w_gu + (size_t)(I + i) * H;
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) {
            g += bf16_value(wg[h]) * x[h];
            u += bf16_value(wu[h]) * x[h];
        }
        a_scratch[i] = silu(s_gu * g) * (s_gu * u);
    }
    for (int h = 0; h < H; ++h) {
        const uint16_t* wd = w_d + (size_t)h * I;
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += bf16_value(wd[i]) * a_scratch[i];
        y[h] = s_d * acc;
    }
}

/*
 * The whole layer for a list of tokens.
 *
 *   hidden     [T, H]      bf16 bits
 *   logits     [T, E]      fp32
 *   w_gate_up  [E, 2I, H]  bf16 bits
 *   w_down     [E, H, I]   bf16 bits
 *   ws_gate_up [2I_s, H]   bf16 bits
 *   ws_down    [H, I_s]    bf16 bits
 *   w_g        [H]         bf16 bits
 *   tokens     [n_tok]     token indices to evaluate (NULL: all T, n_tok = T)
 *   gate_override [n_tok]  NULL, or a shared-gate value to use instead of
 *                          sigmoid(x . w_g) (a hook for the gate pins)
 *   scale_gu, scale_d [E]  NULL (1), or the matrix scale of each expert's
 *                          W_gate_up / W_down (NVFP4 weights)
 *   scale_s_gu, scale_s_d  the shared expert's matrix scales (1 for bf16)
 *   out        [n_tok, H]  fp64
 *   ids_out    [n_tok, k]  selected experts (may be NULL)
 *   w_out      [n_tok, k]  renormalised weights (may be NULL)
 *   gate_out   [n_tok]     shared gate value (may be NULL)
 * Tokens are independent; they are spread over n_threads OpenMP threads.
 * Returns the number of tokens whose score order contradicted the logit order.
 */
int oracle_moe_forward(int T, int H, int E, int k, int I, int I_s, int score_fn,
                       const uint16_t* hidden, const float* logits, const uint16_t* w_gate_up,
                       const uint16_t* w_down, const uint16_t* ws_gate_up,
                       const uint16_t* ws_down, const uint16_t* w_g, const int64_t* tokens,
                       int n_tok, const double* gate_override, const double* scale_gu,
                       const double* scale_d, double scale_s_gu, double scale_s_d, double* out,
                       int32_t* ids_out, double* w_out, double* gate_out, int n_threads) {
    if (tokens == NULL) n_tok = T;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads) reduction(+ : bad)
    for (int n = 0; n < n_tok; ++n) {
        int64_t t = tokens ? tokens[n] : n;
        double* x = (double*)malloc(sizeof(double) * (size_t)H);
        double* y = (double*)malloc(sizeof(double) * (size_t)H);
        double* a = (double*)malloc(sizeof(double) * (size_t)(I > I_s ? I : I_s));
        int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
        double* w = (double*)malloc(sizeof(double) * (size_t)k);
        double* o = out + (size_t)n * H;

        for (int h = 0; h < H; ++h) x[h] = bf16_value(hidden[(size_t)t * H + h]);
        if (oracle_route_token(E, k, score_fn, logits + (size_t)t * E, ids, w) != 0) ++bad;

        for (int h = 0; h < H; ++h) o[h] = 0.0;
        /* routed experts, in selection order */
        for (int j = 0; j < k; ++j) {
            int e = ids[j];
            swiglu_ffn(H, I, w_gate_up + (size_t)e * 2 * I * H, w_down + (size_t)e * H * I,
                       scale_gu ? scale_gu[e] : 1.0, scale_d ? scale_d[e] : 1.0, x, a, y);
            for (int h = 0; h < H; ++h) o[h] += w[j] * y[h];
        }
        /* shared expert with its per-token sigmoid gate */
        double gate;
        if (gate_override) {
            gate = gate_override[n];
        } else {
            double s = 0.0;
            for (int h = 0; h < H; ++h) s += bf16_value(w_g[h]) * x[h];
            gate = 1.0 / (1.0 + exp(-s));
        }
        swiglu_ffn(H, I_s, ws_gate_up, ws_down, scale_s_gu, scale_s_d, x, a, y);
        for (int h = 0; h < H; ++h) o[h] += gate * y[h];

        if (ids_out)
            for (int j = 0; j < k; ++j) ids_out[(size_t)n * k + j] = ids[j];
        if (w_out)
            for (int j = 0; j < k; ++j) w_out[(size_t)n * k + j] = w[j];
        if (gate_out) gate_out[n] = gate;
        free(x); free(y); free(a); free(ids); free(w);
    }
    return bad;
}
