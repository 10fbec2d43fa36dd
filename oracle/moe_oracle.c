/*
 * moe_oracle.c -- plain, slow CPU reference for the fused MoE expert layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load this file.  The product path (the
 * CUDA library) shares no code, header, table or constant with it.
 *
 * Every value is decoded exactly to double and every sum is accumulated in
 * double, one routed row at a time, in the order the sources describe the
 * computation.  No blocking, no fusion, no reordering.
 *
 * Sources (by page title and section):
 *   [MK]   vLLM "Fused MoE Modular Kernel" design doc -- Introduction (the
 *          Contiguous (M,K) and Batched (E,max_tokens,K) activation formats),
 *          "apply()" (permute, W1 matmul, act+mul, quantisation, W2 matmul,
 *          unpermute, TopK weight application + reduce), "TopKWeightAndReduce".
 *   [CAKE] FlashInfer PR 5148 analysis "Cake MegaMoE EP16, BF16 activations x
 *          MXFP8 weights" -- section 2 (_interleave_gate_up_16 "After",
 *          _quantize_mxfp8_block32 "After" scale rule), section 3 (FC2 result
 *          written to the (token, top-k slot) buffer, ordered Top-K reduce).
 *   [MEGA] transformers PR 49606 analysis "DeepGEMM Mega MoE as an EP
 *          implementation" -- section 2 (padding slots: expert id -1, weight 0,
 *          skipped by the kernel).
 *   [DET]  FlashInfer PR 9132 analysis "Cake deterministic MoE grouped GEMM"
 *          -- empty groups give +0.0 (never -0.0).
 *   [OCP]  OCP Microscaling (MX) v1.0 / OFP8 format definitions: E4M3
 *          (bias 7, no infinities, max 448, subnormals), E8M0 (2^(code-127)).
 *
 * Readings where the sources are silent or disagree (each is listed with its
 * reason in the design notes):
 *   - Routing is softmax over all E logits, top-k, then renormalisation of the
 *     chosen k; this equals a softmax over the chosen k logits, so selection is
 *     made on the logits themselves (ties: lower expert index wins).
 *   - W1 of expert e holds 2I rows.  Layout 0: rows [0,I) are gate, [I,2I) up.
 *     Layout 1 ([CAKE] _interleave_gate_up_16 "After"): rows come in groups of
 *     32, the first 16 are gate rows, the next 16 the matching up rows.
 *     h = silu(gate) * up.
 *   - MXFP8 scale code = clamp(c + 127, 0, 254) with c the smallest integer
 *     such that blockmax <= 448 * 2^c (the exact value of ceil(log2(max/448)));
 *     code 0 when the block is all zero.  Blocks run along the contraction
 *     dimension (K for W1, I for W2).
 *   - E4M3 encoding: round to nearest even, saturate to +-448, sign of zero
 *     kept.
 *   - Quantised activations (optional): x rows are MXFP8-quantised along K
 *     from their stored values; h is rounded to the element type its producer
 *     stores (binary32 or bfloat16) before its MXFP8 quantisation along I, so
 *     that a code is decided from the same value on both sides.
 *
 * Parity unpinned: nothing here; see the tests for each pin.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_EXPORT __attribute__((visibility("default")))

/* Element types understood by the oracle (its own numbering). */
enum { OR_F32 = 0, OR_BF16 = 1, OR_E4M3 = 2, OR_F64 = 3 };

/* Error bits reported by the oracle. */
enum { OR_ERR_ID_RANGE = 1, OR_ERR_CAPACITY = 2, OR_ERR_BAD_ARG = 256 };

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* bfloat16 is the upper half of an IEEE binary32. */
ORACLE_EXPORT double oracle_bf16_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round a finite double to the nearest value that has at most `p` significant
 * bits and whose exponent is not below `emin` (values below 2^emin are on the
 * fixed grid 2^(emin-p+1), i.e. IEEE subnormals).  Ties go to even.
 * Division and multiplication by a power of two are exact here.
 */
static double round_to_grid(double v, int p, int emin) {
    if (v == 0.0 || !isfinite(v)) return v;
    int e2;
    frexp(fabs(v), &e2);          /* |v| = m * 2^e2, m in [0.5, 1) */
    int lead = e2 - 1;            /* exponent of the leading bit */
    if (lead < emin) lead = emin;
    double quantum = ldexp(1.0, lead - (p - 1));
    double r = nearbyint(v / quantum) * quantum;   /* default mode: ties-to-even */
    if (r == 0.0) r = copysign(0.0, v);
    return r;
}

/* binary32: 24 significant bits, min normal exponent -126. */
ORACLE_EXPORT float oracle_round_f32(double v) {
    double r = round_to_grid(v, 24, -126);
    if (fabs(r) > 3.4028234663852886e38) return (float)copysign(INFINITY, v);
    return (float)r;
}

/* bfloat16: 8 significant bits, same exponent range as binary32. */
ORACLE_EXPORT uint16_t oracle_double_to_bf16(double v) {
    if (isnan(v)) return 0x7FC0;
    double r = round_to_grid(v, 8, -126);
    float f;
    if (fabs(r) > 3.3895313892515355e38)   /* largest finite bf16 */
        f = (float)copysign(INFINITY, v);
    else
        f = (float)r;                       /* exact: r fits in binary32 */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* E4M3 ([OCP]): s eeee mmm, bias 7; e=0 subnormal m*2^-9; 0x7F/0xFF NaN. */
ORACLE_EXPORT double oracle_e4m3_to_double(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Nearest E4M3 value (ties to even), saturating to +-448, sign kept. */
ORACLE_EXPORT uint8_t oracle_double_to_e4m3(double v) {
    uint8_t sign = (v < 0.0 || (v == 0.0 && signbit(v))) ? 0x80 : 0x00;
    double r = fabs(round_to_grid(v, 4, -6));   /* 4 significant bits, emin -6 */
    if (r > 448.0) r = 448.0;                    /* saturate */
    if (r == 0.0) return sign;
    int e2;
    frexp(r, &e2);
    int lead = e2 - 1;
    if (lead < -6) {                             /* subnormal: m * 2^-9 */
        int m = (int)ldexp(r, 9);
        return sign | (uint8_t)m;
    }
    int m = (int)ldexp(r, 3 - lead) - 8;         /* r = (1 + m/8) 2^lead */
    return sign | (uint8_t)((lead + 7) << 3) | (uint8_t)m;
}

/* E8M0 scale: 2^(code-127); 255 is NaN. */
ORACLE_EXPORT double oracle_e8m0_to_double(uint8_t code) {
    if (code == 255) return NAN;
    return ldexp(1.0, (int)code - 127);
}

/*
 * [CAKE] section 2, _quantize_mxfp8_block32 "After": the scale code of a block
 * of 32 is clamp(ceil(log2(max/448)) + 127, 0, 254), and 0 when the block is
 * all zero.  ceil(log2(m/448)) is the smallest integer c with m <= 448*2^c;
 * both sides of that comparison are exact doubles.
 */
ORACLE_EXPORT uint8_t oracle_mxfp8_scale_code(double blockmax) {
    if (!(blockmax > 0.0)) return 0;
    int c;
    frexp(blockmax / 448.0, &c);          /* 2^(c-1) <= m/448 < 2^c (approx) */
    while (blockmax > ldexp(448.0, c)) c++;
    while (blockmax <= ldexp(448.0, c - 1)) c--;
    int code = c + 127;
    if (code < 0) code = 0;
    if (code > 254) code = 254;
    return (uint8_t)code;
}

static double load_elem(const void* p, int dtype, int64_t idx) {
    switch (dtype) {
    case OR_F32: return (double)((const float*)p)[idx];
    case OR_BF16: return oracle_bf16_to_double(((const uint16_t*)p)[idx]);
    case OR_E4M3: return oracle_e4m3_to_double(((const uint8_t*)p)[idx]);
    case OR_F64: return ((const double*)p)[idx];
    }
    return NAN;
}

static void store_elem(void* p, int dtype, int64_t idx, double v) {
    switch (dtype) {
    case OR_F32: ((float*)p)[idx] = oracle_round_f32(v); break;
    case OR_BF16: ((uint16_t*)p)[idx] = oracle_double_to_bf16(v); break;
    case OR_E4M3: ((uint8_t*)p)[idx] = oracle_double_to_e4m3(v); break;
    case OR_F64: ((double*)p)[idx] = v; break;
    }
}

/*
 * MXFP8 block-32 quantisation of a (rows, cols) matrix, blocks of 32
 * consecutive elements along each row ([CAKE] section 2; [OCP]).
 * codes: (rows, cols) E4M3; scales: (rows, cols/32) E8M0.
 * Returns 0, or -1 when cols is not a multiple of 32.
 */
ORACLE_EXPORT int oracle_mxfp8_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols,
                                        uint8_t* codes, uint8_t* scales) {
    if (cols % 32 != 0) return -1;
    int64_t nb = cols / 32;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            double m = 0.0;
            for (int i = 0; i < 32; ++i) {
                double a = fabs(load_elem(x, x_dtype, r * cols + b * 32 + i));
                if (a > m) m = a;
            }
            uint8_t code = oracle_mxfp8_scale_code(m);
            scales[r * nb + b] = code;
            double scale = oracle_e8m0_to_double(code);
            for (int i = 0; i < 32; ++i) {
                double v = load_elem(x, x_dtype, r * cols + b * 32 + i);
                codes[r * cols + b * 32 + i] = oracle_double_to_e4m3(v / scale);
            }
        }
    }
    return 0;
}

/*
 * Decode MXFP8: out[r, c] = E4M3(codes[r, c]) * 2^(scales[r, c/32] - 127).
 */
ORACLE_EXPORT int oracle_mxfp8_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols,
                                          double* out) {
    if (cols % 32 != 0) return -1;
    int64_t nb = cols / 32;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            out[r * cols + c] = oracle_e4m3_to_double(codes[r * cols + c]) * oracle_e8m0_to_double(scales[r * nb + c / 32]);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Routing                                                                   */
/* ------------------------------------------------------------------------ */

/*
 * Top-k routing (the "select_experts" step named in [MK], How-To, topk
 * indices dtype): per token, the k largest logits (ties: lower index first),
 * weights p_j = exp(l_j - l_max) normalised over the chosen k (renormalize=1)
 * or over all E experts (renormalize=0, plain softmax probabilities).
 */
ORACLE_EXPORT int oracle_topk_route(const float* logits, int64_t T, int E, int k, int renormalize,
                                    int32_t* ids, float* weights) {
    if (k < 1 || k > E) return -1;
    char* taken = (char*)malloc((size_t)E);
    if (!taken) return -2;
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;   /* strict: lower index keeps ties */
            }
            taken[best] = 1;
            ids[t * k + j] = best;
        }
        double lmax = (double)l[ids[t * k]];
        double denom = 0.0;
        if (renormalize) {
            for (int j = 0; j < k; ++j) denom += exp((double)l[ids[t * k + j]] - lmax);
        } else {
            for (int e = 0; e < E; ++e) denom += exp((double)l[e] - lmax);
        }
        for (int j = 0; j < k; ++j)
            weights[t * k + j] = oracle_round_f32(exp((double)l[ids[t * k + j]] - lmax) / denom);
    }
    free(taken);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Permute / align                                                           */
/* ------------------------------------------------------------------------ */

/*
 * Contiguous layout ([MK] Introduction and apply(): Permute).  Route r = t*k+j
 * goes to expert ids[r]; -1 is a padding slot and is skipped ([MEGA] sec. 2);
 * an id outside [-1, E) sets OR_ERR_ID_RANGE and is skipped.
 *   counts[e]          routes of expert e
 *   offsets[e+1]       offsets[e] + ceil(counts[e]/block_m)*block_m
 *   sorted_route[s]    the route placed in row s, rows of an expert filled in
 *                      increasing route index; -1 in padding rows
 *   route_row[r]       the row of route r, or -1
 * sorted_route must hold offsets[E] entries (at most T*k + E*(block_m-1)).
 * Returns the error bits.
 */
ORACLE_EXPORT int oracle_permute_contiguous(const int32_t* ids, int64_t T, int k, int E, int block_m,
                                            int32_t* counts, int32_t* offsets, int32_t* sorted_route,
                                            int32_t* route_row) {
    if (E <= 0 || k <= 0 || block_m <= 0 || T < 0) return OR_ERR_BAD_ARG;
    int err = 0;
    int64_t R = T * k;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t r = 0; r < R; ++r) {
        int e = ids[r];
        if (e == -1) continue;
        if (e < -1 || e >= E) { err |= OR_ERR_ID_RANGE; continue; }
        counts[e]++;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        int padded = (counts[e] + block_m - 1) / block_m * block_m;
        offsets[e + 1] = offsets[e] + padded;
    }
    for (int64_t s = 0; s < offsets[E]; ++s) sorted_route[s] = -1;
    int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int64_t r = 0; r < R; ++r) {
        int e = ids[r];
        route_row[r] = -1;
        if (e < 0 || e >= E) continue;
        int64_t s = offsets[e] + fill[e]++;
        sorted_route[s] = (int32_t)r;
        route_row[r] = (int32_t)s;
    }
    free(fill);
    return err;
}

/*
 * Batched layout ([MK] Introduction: (num_experts, max_tokens, K) plus
 * expert_num_tokens).  Route r becomes row (e, rank) where rank counts the
 * earlier routes of expert e.  Ranks >= max_tokens do not fit: their routes
 * are dropped and OR_ERR_CAPACITY is set (the routing-capacity validation
 * named in [CAKE] "Why is this good?", item 4).  expert_num_tokens[e] = min(count, max).
 * row_route has E*max_tokens entries: the route of each row, or -1.
 */
ORACLE_EXPORT int oracle_permute_batched(const int32_t* ids, int64_t T, int k, int E, int max_tokens,
                                         int32_t* expert_num_tokens, int32_t* row_route,
                                         int32_t* route_row) {
    if (E <= 0 || k <= 0 || max_tokens < 0 || T < 0) return OR_ERR_BAD_ARG;
    int err = 0;
    int64_t R = T * k;
    for (int e = 0; e < E; ++e) expert_num_tokens[e] = 0;
    for (int64_t s = 0; s < (int64_t)E * max_tokens; ++s) row_route[s] = -1;
    int32_t* rank = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int64_t r = 0; r < R; ++r) {
        int e = ids[r];
        route_row[r] = -1;
        if (e == -1) continue;
        if (e < -1 || e >= E) { err |= OR_ERR_ID_RANGE; continue; }
        int q = rank[e]++;
        if (q >= max_tokens) { err |= OR_ERR_CAPACITY; continue; }
        int64_t s = (int64_t)e * max_tokens + q;
        row_route[s] = (int32_t)r;
        route_row[r] = (int32_t)s;
        expert_num_tokens[e] = q + 1;
    }
    free(rank);
    return err;
}

/* ------------------------------------------------------------------------ */
/* Expert FFN                                                                */
/* ------------------------------------------------------------------------ */

/* Row of W1[e] that holds gate (half=0) or up (half=1) unit i. */
static int64_t w1_row(int w1_layout, int64_t I, int half, int64_t i) {
    if (w1_layout == 0) return half * I + i;              /* [gate; up] */
    return (i / 16) * 32 + half * 16 + (i % 16);           /* gate16, up16, ... */
}

/* Weight element (row, col) of an (rows, cols) matrix, MXFP8-decoded if E4M3. */
static double weight_elem(const void* w, int w_dtype, const uint8_t* w_scale, int64_t base_elem,
                          int64_t row, int64_t col, int64_t cols) {
    double v = load_elem(w, w_dtype, base_elem + row * cols + col);
    if (w_dtype == OR_E4M3) {
        int64_t scale_idx = base_elem / 32 + row * (cols / 32) + col / 32;
        v *= oracle_e8m0_to_double(w_scale[scale_idx]);
    }
    return v;
}

static double silu(double g) { return g / (1.0 + exp(-g)); }

/*
 * [MK] apply(): "Matmul with W1" then "Act + Mul", one routed row at a time.
 * x row r (K elements of x_dtype) goes through expert row_expert[r]:
 *   g_i = sum_k x[k] W1[e, gate_row(i), k],  u_i likewise,  h_i = silu(g_i)*u_i.
 * W1: (E, 2I, K).  Rows with expert -1 give h = 0.  h: (nrows, I) in h_dtype.
 */
ORACLE_EXPORT int oracle_expert_gate_up(const void* x, int x_dtype, int64_t nrows, const int32_t* row_expert,
                                        const void* w1, const uint8_t* w1_scale, int w_dtype, int w1_layout,
                                        int E, int64_t K, int64_t I, void* h, int h_dtype) {
    for (int64_t r = 0; r < nrows; ++r) {
        int e = row_expert[r];
        for (int64_t i = 0; i < I; ++i) {
            double hv = 0.0;
            if (e >= 0 && e < E) {
                int64_t base = (int64_t)e * 2 * I * K;
                int64_t rg = w1_row(w1_layout, I, 0, i), ru = w1_row(w1_layout, I, 1, i);
                double g = 0.0, u = 0.0;
                for (int64_t c = 0; c < K; ++c) {
                    double xv = load_elem(x, x_dtype, r * K + c);
                    g += xv * weight_elem(w1, w_dtype, w1_scale, base, rg, c, K);
                    u += xv * weight_elem(w1, w_dtype, w1_scale, base, ru, c, K);
                }
                hv = silu(g) * u;
            }
            store_elem(h, h_dtype, r * I + i, hv);
        }
    }
    return 0;
}

/*
 * [MK] apply(): "Matmul with W2".  y_n = sum_i h[i] W2[e, n, i];
 * W2: (E, K, I).  Rows with expert -1 give y = 0.  y: (nrows, K).
 */
ORACLE_EXPORT int oracle_expert_down(const void* h, int h_dtype, int64_t nrows, const int32_t* row_expert,
                                     const void* w2, const uint8_t* w2_scale, int w_dtype,
                                     int E, int64_t K, int64_t I, void* y, int y_dtype) {
    for (int64_t r = 0; r < nrows; ++r) {
        int e = row_expert[r];
        for (int64_t n = 0; n < K; ++n) {
            double acc = 0.0;
            if (e >= 0 && e < E) {
                int64_t base = (int64_t)e * K * I;
                for (int64_t i = 0; i < I; ++i)
                    acc += load_elem(h, h_dtype, r * I + i) * weight_elem(w2, w_dtype, w2_scale, base, n, i, I);
            }
            store_elem(y, y_dtype, r * K + n, acc);
        }
    }
    return 0;
}

/*
 * [MK] TopKWeightAndReduce (Contiguous); [CAKE] section 3 ordered Top-K
 * reduce.  y_slots: (T, k, K), the expert output of each (token, slot).
 *   out[t] = sum over j = 0..k-1 with ids[t,j] != -1 of w[t,j] * y_slots[t,j]
 * in increasing j.  weights may be NULL (already applied).  A token whose
 * slots are all padding gets +0.0 ([DET] empty groups).
 */
ORACLE_EXPORT int oracle_topk_reduce(const void* y_slots, int y_dtype, const int32_t* ids, const float* weights,
                                     int64_t T, int k, int64_t K, void* out, int out_dtype) {
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t n = 0; n < K; ++n) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                if (ids[t * k + j] < 0) continue;
                double w = weights ? (double)weights[t * k + j] : 1.0;
                acc += w * load_elem(y_slots, y_dtype, (t * k + j) * K + n);
            }
            store_elem(out, out_dtype, t * K + n, acc);
        }
    }
    return 0;
}

/*
 * [MK] TopKWeightAndReduce for the Batched format (NaiveBatched), taken all
 * the way to token order: the expert outputs sit in rows (e, q) of an
 * (E, max_tokens, K) buffer, seen here as `rows` rows of K, and route_row maps
 * each route r = t*k + j to its row (-1: padding or dropped for capacity).
 *   out[t] = sum over j = 0..k-1 with route_row[t*k+j] != -1 of
 *            w[t,j] * y_rows[route_row[t*k+j]]
 * in increasing j, from +0.0.  Rows outside [-1, rows) are skipped and
 * reported as OR_ERR_ID_RANGE.
 */
ORACLE_EXPORT int oracle_batched_topk_reduce(const void* y_rows, int y_dtype, int64_t rows, const int32_t* route_row,
                                             const float* weights, int64_t T, int k, int64_t K, void* out,
                                             int out_dtype) {
    int err = 0;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t n = 0; n < K; ++n) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                int64_t row = route_row[t * k + j];
                if (row == -1) continue;
                if (row < -1 || row >= rows) { err |= OR_ERR_ID_RANGE; continue; }
                double w = weights ? (double)weights[t * k + j] : 1.0;
                acc += w * load_elem(y_rows, y_dtype, row * K + n);
            }
            store_elem(out, out_dtype, t * K + n, acc);
        }
    }
    return err;
}

/*
 * One routed row through the whole expert: optional MXFP8 quantisation of the
 * activation row ([MK] "prepare": input activation quantisation; block 32
 * along K, then decoded), gate/up, act*mul, optional MXFP8 quantisation of h
 * ([MK] apply(): "Quantisation" between act+mul and W2; h is first rounded to
 * the precision the producer stores it in -- quant_h = 1: binary32,
 * quant_h = 2: bfloat16 -- then block-32 quantised along I and decoded), down.
 */
static void expert_ffn_row(const void* xrow, int x_dtype, int e,
                           const void* w1, const uint8_t* w1_scale, const void* w2, const uint8_t* w2_scale,
                           int w_dtype, int w1_layout, int E, int64_t K, int64_t I, int quant_x, int quant_h,
                           double* h, double* y) {
    int32_t one_expert = e;
    if (quant_x) {
        uint8_t* codes = (uint8_t*)malloc((size_t)K);
        uint8_t* scales = (uint8_t*)malloc((size_t)(K / 32));
        double* xq = (double*)malloc(sizeof(double) * (size_t)K);
        oracle_mxfp8_quantize(xrow, x_dtype, 1, K, codes, scales);
        oracle_mxfp8_dequantize(codes, scales, 1, K, xq);
        oracle_expert_gate_up(xq, OR_F64, 1, &one_expert, w1, w1_scale, w_dtype, w1_layout, E, K, I, h, OR_F64);
        free(codes); free(scales); free(xq);
    } else {
        oracle_expert_gate_up(xrow, x_dtype, 1, &one_expert, w1, w1_scale, w_dtype, w1_layout, E, K, I, h, OR_F64);
    }
    if (quant_h) {
        void* hs;
        int hs_dtype;
        if (quant_h == 2) {
            uint16_t* hb = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
            for (int64_t i = 0; i < I; ++i) hb[i] = oracle_double_to_bf16(h[i]);
            hs = hb;
            hs_dtype = OR_BF16;
        } else {
            float* hf = (float*)malloc(sizeof(float) * (size_t)I);
            for (int64_t i = 0; i < I; ++i) hf[i] = oracle_round_f32(h[i]);
            hs = hf;
            hs_dtype = OR_F32;
        }
        uint8_t* codes = (uint8_t*)malloc((size_t)I);
        uint8_t* scales = (uint8_t*)malloc((size_t)(I / 32));
        oracle_mxfp8_quantize(hs, hs_dtype, 1, I, codes, scales);
        oracle_mxfp8_dequantize(codes, scales, 1, I, h);
        free(hs); free(codes); free(scales);
    }
    oracle_expert_down(h, OR_F64, 1, &one_expert, w2, w2_scale, w_dtype, E, K, I, y, OR_F64);
}

/*
 * The whole contiguous layer ([MK] apply() followed by TopKWeightAndReduce):
 * for each token t and slot j with expert e = ids[t,j] != -1,
 *   y = FFN_e(x[t]),  out[t] += w[t,j] * y   (j increasing, from +0.0).
 * x: (T, K); out: (T, K) of out_dtype.  Ids outside [-1, E) are skipped and
 * reported.  Returns the error bits.
 */
ORACLE_EXPORT int oracle_moe_layer(const void* x, int x_dtype, int64_t T, int64_t K, int64_t I, int E, int k,
                                   const int32_t* ids, const float* weights,
                                   const void* w1, const uint8_t* w1_scale, const void* w2, const uint8_t* w2_scale,
                                   int w_dtype, int w1_layout, int quant_x, int quant_h, void* out, int out_dtype) {
    int err = 0;
    double* h = (double*)malloc(sizeof(double) * (size_t)I);
    double* y = (double*)malloc(sizeof(double) * (size_t)K);
    double* acc = (double*)malloc(sizeof(double) * (size_t)K);
    int esz = x_dtype == OR_F32 ? 4 : (x_dtype == OR_BF16 ? 2 : (x_dtype == OR_F64 ? 8 : 1));
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t n = 0; n < K; ++n) acc[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            int e = ids[t * k + j];
            if (e == -1) continue;
            if (e < -1 || e >= E) { err |= OR_ERR_ID_RANGE; continue; }
            const char* xrow = (const char*)x + (size_t)(t * K) * esz;
            expert_ffn_row(xrow, x_dtype, e, w1, w1_scale, w2, w2_scale, w_dtype, w1_layout, E, K, I, quant_x, quant_h,
                           h, y);
            double w = weights ? (double)weights[t * k + j] : 1.0;
            for (int64_t n = 0; n < K; ++n) acc[n] += w * y[n];
        }
        for (int64_t n = 0; n < K; ++n) store_elem(out, out_dtype, t * K + n, acc[n]);
    }
    free(h); free(y); free(acc);
    return err;
}

/*
 * The batched layer with the naive-batched weight application ([MK]
 * TopKWeightAndReduceNaiveBatched, read as a per-row weight in place):
 *   out[e, r] = w[e, r] * FFN_e(xb[e, r])  for r < expert_num_tokens[e].
 * xb: (E, max_tokens, K); w: (E, max_tokens) or NULL; out: (E, max_tokens, K).
 * Rows r >= expert_num_tokens[e] are neither read nor written.
 */
ORACLE_EXPORT int oracle_moe_layer_batched(const void* xb, int x_dtype, int E, int64_t max_tokens,
                                           const int32_t* expert_num_tokens, const float* weights,
                                           int64_t K, int64_t I,
                                           const void* w1, const uint8_t* w1_scale, const void* w2,
                                           const uint8_t* w2_scale, int w_dtype, int w1_layout, int quant_x,
                                           int quant_h, void* out, int out_dtype) {
    double* h = (double*)malloc(sizeof(double) * (size_t)I);
    double* y = (double*)malloc(sizeof(double) * (size_t)K);
    int esz = x_dtype == OR_F32 ? 4 : (x_dtype == OR_BF16 ? 2 : (x_dtype == OR_F64 ? 8 : 1));
    int err = 0;
    for (int e = 0; e < E; ++e) {
        int64_t cnt = expert_num_tokens[e];
        if (cnt < 0 || cnt > max_tokens) { err |= OR_ERR_CAPACITY; continue; }
        for (int64_t r = 0; r < cnt; ++r) {
            int64_t row = (int64_t)e * max_tokens + r;
            const char* xrow = (const char*)xb + (size_t)(row * K) * esz;
            expert_ffn_row(xrow, x_dtype, e, w1, w1_scale, w2, w2_scale, w_dtype, w1_layout, E, K, I, quant_x, quant_h,
                           h, y);
            double w = weights ? (double)weights[row] : 1.0;
            for (int64_t n = 0; n < K; ++n) store_elem(out, out_dtype, row * K + n, w * y[n]);
        }
    }
    free(h); free(y);
    return err;
}
