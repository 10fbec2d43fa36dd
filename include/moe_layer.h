/*
 * moe_layer.h -- C ABI of the GB300 fused MoE expert layer (libmoe_layer.so).
 *
 * The layer is six calls issued in order on one CUDA stream:
 *
 *   moe_topk_route -> moe_permute_align -> moe_gemm1_swiglu
 *     -> (optional) mxfp8_quantize_block32 -> moe_gemm2
 *     -> moe_unpermute_topk_reduce | moe_batched_weight_reduce
 *
 * following the decomposition of the vLLM design doc "Fused MoE Modular
 * Kernel", section "apply()": Permute, Matmul with W1, Act + Mul,
 * Quantisation, Matmul with W2, Unpermute, TopK weight application + reduce.
 * Two calls stand for pairs of those steps where one launch serves better:
 * moe_route_permute_align (routing + placement + row gather; one launch for
 * decode-sized batches) and moe_experts_fused (both GEMMs in one launch, the
 * decode regime).  moe_batched_topk_reduce combines batched rows into token
 * order.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every array argument is a DEVICE pointer to caller-owned memory.  The
 *   library never allocates, frees or synchronises; it only launches kernels
 *   on `stream` (a cudaStream_t passed as void*; NULL = the legacy default
 *   stream).  All calls are asynchronous.
 * - Matrices are row-major and dense (the last index is contiguous).
 * - Element types: MOE_F32 (binary32), MOE_BF16 (bfloat16), MOE_E4M3
 *   (OCP E4M3FN codes, one byte each, always paired with one E8M0 scale byte
 *   per 32 consecutive elements along the contraction dimension).  The E4M3
 *   NaN codes 0x7F and 0xFF, and the E8M0 NaN scale 0xFF, are outside the
 *   contract: mxfp8_quantize_block32 never writes them (it saturates, and its
 *   largest scale is 254), and a GEMM given them returns unspecified values
 *   without an error bit (the bf16-activation path decodes 0x7F/0xFF as the
 *   finite value 480 * scale, where the format defines NaN).
 * - Expert ids are int32; -1 marks a padding slot that every step skips
 *   (transformers PR 49606 analysis "DeepGEMM Mega MoE as an EP
 *   implementation", section 2: padded slots carry expert id -1, weight 0).
 * - Return value: MOE_OK, or an error status found on the host before any
 *   launch (nothing is launched then).  moe_last_error() gives a message for
 *   the calling thread's last failure.
 * - Errors that depend on device data never trap.  Kernels OR bits into
 *   *err_word (a device int32 the caller zeroes and reads when it likes;
 *   err_word may be NULL where documented): MOE_DEVERR_ID_RANGE for an id
 *   outside [-1, E), MOE_DEVERR_CAPACITY for a batched expert over capacity,
 *   MOE_DEVERR_TIMEOUT when a pipeline wait inside a GEMM gave up (the
 *   kernel then returns early and its outputs are unspecified).
 * - Sizes are int64 where they can exceed 2^31 elements.
 * - Test hook: when the environment variable MOE_TEST_SKIP_FIRST_COPY is "1"
 *   at the first tcgen05 GEMM launch of the process, CTA 0 of every tcgen05
 *   GEMM leaves its first stage's copy out, so that stage never fills and
 *   the kernel reports MOE_DEVERR_TIMEOUT after 2 s (its outputs are then
 *   unspecified).  It exists to test the bounded waits without a fault;
 *   never set it in production.
 */
#ifndef MOE_LAYER_H
#define MOE_LAYER_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (host) ---- */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1         /* null pointer, bad size or enum */
#define MOE_ERR_UNSUPPORTED 2         /* dtype/layout combination, or no sm_103a device */
#define MOE_ERR_ALIGNMENT 3           /* pointer or row pitch not 16-byte aligned, or a size not a multiple of 32 */
#define MOE_ERR_WORKSPACE_TOO_SMALL 4
#define MOE_ERR_LAUNCH 5              /* a CUDA runtime call failed */

/* ---- device error bits (OR-ed into *err_word) ---- */
#define MOE_DEVERR_ID_RANGE 1
#define MOE_DEVERR_CAPACITY 2
#define MOE_DEVERR_TIMEOUT 4
#define MOE_DEVERR_INTERNAL 8         /* a kernel's own consistency check failed (the two CTAs of a pair saw
                                         different tensor-memory addresses); it did no work, outputs unspecified */

/* ---- element types ---- */
#define MOE_F32 0
#define MOE_BF16 1
#define MOE_E4M3 2

/* ---- activation layouts ("Fused MoE Modular Kernel", Introduction) ---- */
#define MOE_LAYOUT_CONTIGUOUS 0       /* (M, K) rows grouped by expert */
#define MOE_LAYOUT_BATCHED 1          /* (E, max_tokens, K) + expert_num_tokens[E] */

/* ---- W1 row layouts ---- */
#define MOE_W1_GATE_UP 0              /* W1[e] = [gate rows 0..I-1 ; up rows 0..I-1] */
#define MOE_W1_INTERLEAVE16 1         /* rows in groups of 32: 16 gate rows then the 16 matching up rows
                                         ("Cake MegaMoE EP16" FlashInfer PR 5148 analysis, section 2,
                                         _interleave_gate_up_16 "After") */
#define MOE_W_TILED 2                 /* tile-contiguous layout written by moe_tile_weights: W1 and W2 of
                                         moe_experts_fused, W1 of moe_gemm1_swiglu / W2 of moe_gemm2 on
                                         CTA-pair tiles (bf16) or on swap-AB tiles (E4M3 codes) */

/* ---- GEMM implementations ---- */
#define MOE_IMPL_AUTO 0               /* swap-AB tiles when routes/expert are few, else CTA-pair tiles
                                         (bf16; normal tiles for shapes outside them); E4M3 weights on
                                         swap-AB tiles; CUDA cores for fp32 */
#define MOE_IMPL_TCGEN05 1            /* tcgen05 tiles, tokens on the MMA M side (128 rows per tile; 256,
                                         as two MMA halves, for the batched layout) */
#define MOE_IMPL_TCGEN05_SWAP_AB 2    /* tcgen05 tiles, weight rows on the MMA M side, tokens on N
                                         (AWS blog "MoE kernel engineering on SageMaker AI", Swap-AB:
                                         C^T = B^T A^T when M < 64) */
#define MOE_IMPL_SIMT 3               /* CUDA-core FMA tiles (fp32 path, any shape) */
#define MOE_IMPL_TCGEN05_MIXED 4      /* tcgen05: 128-row tiles for experts of 64 rows or more and a swap-AB
                                         tile for each smaller expert, in one launch (bf16 weights) */
#define MOE_IMPL_TCGEN05_PAIR 5       /* tcgen05 on CTA pairs (cta_group::2, two SMs per tile): 256 weight rows
                                         on the MMA M side (128 staged by each SM), up to 256 tokens on N;
                                         bf16 activations and weights, 2I % 256 == 0 (GEMM 1), K % 256 == 0
                                         (GEMM 2), contraction % 64 == 0 */

/* Message describing the calling thread's last failed call ("" if none). */
MOE_API const char* moe_last_error(void);

/* Library version, (major << 16) | minor. */
MOE_API int moe_version(void);

/* Upper bound on the rows of the contiguous layout:
 * T*top_k + E*(block_m - 1) = max over routings of sum_e ceil(count_e/block_m)*block_m.
 * -1 for arguments the permute calls reject (T < 0, top_k or E outside [1, 1024], block_m outside
 * [1, 4096], or T*top_k >= 2^31, which is tested without forming the product). */
MOE_API int64_t moe_max_padded_rows(int64_t T, int top_k, int E, int block_m);

/* Bytes of scratch moe_permute_align needs for T tokens, top_k slots, E experts
 * (the two workspaces declared up front in "Fused MoE Modular Kernel",
 * workspace_shapes()).  0 for arguments the permute calls reject (as for
 * moe_max_padded_rows). */
MOE_API size_t moe_permute_workspace_size(int64_t T, int top_k, int E);

/*
 * moe_topk_route -- per token, the top_k largest of E router logits and their
 * weights.  The weights are softmax over all E, restricted to the chosen
 * experts and renormalised to sum 1 (renormalize != 0), or the plain softmax
 * probabilities (renormalize == 0).  Selection compares the fp32 logits
 * (softmax is monotone); ties go to the lower expert index.
 * ("Fused MoE Modular Kernel", How-To: select_experts and the TopK ids dtype.)
 *
 *   logits        (T, E) fp32
 *   topk_ids      (T, top_k) int32 out, in decreasing logit order
 *   topk_weights  (T, top_k) fp32 out
 * Limits: 1 <= top_k <= min(E, 32), E <= 1024.  T may be 0 (no launch).
 */
MOE_API int moe_topk_route(const float* logits, int64_t T, int E, int top_k, int renormalize,
                   int32_t* topk_ids, float* topk_weights, void* stream);

/*
 * moe_permute_align -- groups the routes r = t*top_k + j into expert-major
 * rows ("Fused MoE Modular Kernel", apply(): Permute; Introduction: the
 * Contiguous and Batched formats).  Within an expert, rows follow increasing
 * route index (a stable order), so the result is unique.
 *
 *   topk_ids        (T, top_k) int32; -1 = padding, skipped; other ids
 *                   outside [0, E) set MOE_DEVERR_ID_RANGE and are skipped.
 *   layout          MOE_LAYOUT_CONTIGUOUS:
 *                     expert_counts[e]   = routes of expert e
 *                     expert_offsets[e]  = sum_{e'<e} ceil(count_e'/block_m)*block_m, E+1 entries
 *                     row_route[s]       = the route in row s, -1 in padding rows; rows_cap entries,
 *                                          entries at and beyond expert_offsets[E] are not written
 *                     rows_cap >= moe_max_padded_rows(T, top_k, E, block_m)
 *                   MOE_LAYOUT_BATCHED (rows (e, q) at e*max_tokens + q):
 *                     expert_counts[e]   = expert_num_tokens[e] = min(count_e, max_tokens);
 *                                          routes beyond max_tokens are dropped and set
 *                                          MOE_DEVERR_CAPACITY
 *                     expert_offsets[e]  = e*max_tokens, E+1 entries
 *                     row_route[s]       = route or -1, all E*max_tokens entries written
 *                     rows_cap == E*max_tokens; block_m is ignored
 *   route_row       (T*top_k) int32 out: the row of each route, -1 for skipped ones
 *   x, x_dtype, K   optional (x may be NULL): (T, K) activations (F32 or BF16) to
 *                   gather into x_out (rows_cap, K); rows holding no route are not written.
 *                   K*element size must be a multiple of 16 bytes.
 *   workspace       >= moe_permute_workspace_size(T, top_k, E) bytes, 256-byte aligned;
 *                   its contents on entry do not matter.
 *   err_word        device int32, may be NULL.
 */
MOE_API int moe_permute_align(const int32_t* topk_ids, int64_t T, int top_k, int E,
                      int layout, int block_m, int max_tokens,
                      const void* x, int x_dtype, int64_t K, void* x_out, int64_t rows_cap,
                      int32_t* expert_counts, int32_t* expert_offsets,
                      int32_t* row_route, int32_t* route_row,
                      void* workspace, size_t workspace_bytes, int32_t* err_word, void* stream);

/*
 * moe_route_permute_align -- moe_topk_route followed by moe_permute_align on
 * the ids it writes ("Fused MoE Modular Kernel", apply(): select_experts, then
 * Permute): same arguments, same results bit for bit, same errors.  For
 * decode-sized batches (T <= 128 and T*top_k <= 1024) the routing, the
 * placement and the gather of x run as one launch, in place of the three
 * launches of the separate calls; larger batches take the separate launches.
 *
 *   logits, renormalize, topk_ids, topk_weights   as for moe_topk_route
 *                                                  (topk_ids is written and
 *                                                  then read by the placement)
 *   every other argument                           as for moe_permute_align
 * Limits: those of both calls (1 <= top_k <= min(E, 32), E <= 1024).
 */
MOE_API int moe_route_permute_align(const float* logits, int64_t T, int E, int top_k, int renormalize,
                      int32_t* topk_ids, float* topk_weights,
                      int layout, int block_m, int max_tokens,
                      const void* x, int x_dtype, int64_t K, void* x_out, int64_t rows_cap,
                      int32_t* expert_counts, int32_t* expert_offsets,
                      int32_t* row_route, int32_t* route_row,
                      void* workspace, size_t workspace_bytes, int32_t* err_word, void* stream);

/*
 * moe_permute_align_static -- moe_permute_align for callers that cannot
 * allocate device memory.  The sources describe no such variant; it exists for
 * callers with no allocator to hand: plugins inside a host framework that owns
 * all device memory, request paths where cudaMalloc/cudaFree (which can
 * synchronise the device) are forbidden, or deployments whose memory budget is
 * fixed at start-up.  Arguments and results are those of moe_permute_align,
 * without workspace and workspace_bytes: the scratch is a 2 MiB array built
 * into the library, reserved on every GPU that loads it until the process
 * exits.  This call allocates nothing.
 *   - Routings needing more than 2 MiB of scratch (moe_permute_workspace_size
 *     > 2 MiB, about 450k routes) return MOE_ERR_WORKSPACE_TOO_SMALL.
 *   - The first call in each CUDA context of a device looks up the array's
 *     device address (cudaGetSymbolAddress); make that first call before any
 *     stream capture.  The address is kept for that context only, so after
 *     cudaDeviceReset (or a re-created primary context) the next call looks
 *     it up again -- again outside any capture.
 *   - T, top_k and E are checked before any size is formed: T*top_k < 2^31,
 *     top_k and E in [1, 1024]; otherwise MOE_ERR_INVALID_ARG, nothing read.
 *   - All calls share the one array: calls that overlap on the GPU (other
 *     streams, other host threads) race and must be serialised by the caller.
 */
MOE_API int moe_permute_align_static(const int32_t* topk_ids, int64_t T, int top_k, int E,
                                     int layout, int block_m, int max_tokens,
                                     const void* x, int x_dtype, int64_t K, void* x_out, int64_t rows_cap,
                                     int32_t* expert_counts, int32_t* expert_offsets,
                                     int32_t* row_route, int32_t* route_row, int32_t* err_word, void* stream);

/*
 * moe_gemm1_swiglu -- grouped GEMM with W1 fused with SiLU-and-mul
 * ("Fused MoE Modular Kernel", apply(): Matmul with W1, Act + Mul).
 * For every valid row s of expert e:
 *     g_i = sum_k a[s,k] W1[e, gate_row(i), k],  u_i likewise with up_row(i),
 *     h[s, i] = silu(g_i) * u_i = g_i / (1 + exp(-g_i)) * u_i,   i < I.
 *
 *   a             rows of activations, element type a_dtype (F32, BF16, or E4M3 codes)
 *                   contiguous: (rows_cap, K); expert e owns rows
 *                     [expert_offsets[e], expert_offsets[e] + expert_counts[e])
 *                   batched: (E, max_tokens, K); expert e owns rows [0, expert_counts[e])
 *   a_scale       E4M3 activations ("Fused MoE Modular Kernel", prepare(): input
 *                 activation quantisation, from mxfp8_quantize_block32): E8M0 bytes,
 *                 same rows as `a`, K/32 per row, 4-byte aligned; NULL otherwise.
 *                 E4M3 activations need E4M3 weights and run on block-scaled tcgen05
 *                 swap-AB tiles (K % 128 == 0, 2I % 128 == 0) or MOE_IMPL_SIMT.
 *   w1            (E, 2I, K) of w_dtype (F32, BF16 or E4M3); rows per w1_layout: MOE_W1_GATE_UP,
 *                 MOE_W1_INTERLEAVE16, or MOE_W_TILED (from moe_tile_weights, which = 1: bf16
 *                 weights on CTA-pair tiles, MOE_IMPL_AUTO or MOE_IMPL_TCGEN05_PAIR; E4M3 codes on
 *                 swap-AB tiles, MOE_IMPL_AUTO or MOE_IMPL_TCGEN05_SWAP_AB; else
 *                 MOE_ERR_UNSUPPORTED)
 *   w1_scale      (E, 2I, K/32) E8M0 bytes when w_dtype == MOE_E4M3, else NULL
 *   h             same row indexing as `a`, (rows, I) of h_dtype (F32, BF16, or E4M3 codes);
 *                 only valid rows are written.
 *   h_scale       h_dtype == MOE_E4M3 ("Fused MoE Modular Kernel", apply(): quantisation
 *                 between act+mul and W2, done in this call's epilogue): E8M0 scales of h,
 *                 (rows, I/32), written with h; the codes equal those of
 *                 mxfp8_quantize_block32 applied to the BF16 h this call would otherwise
 *                 write.  NULL for F32/BF16 h.  Block-scaled tcgen05 tiles (E4M3 activations)
 *                 or MOE_IMPL_SIMT.
 *   impl          MOE_IMPL_*; the tcgen05 paths need BF16 activations, BF16 or E4M3
 *                 weights, K % 64 == 0 and I % 64 == 0 (MOE_ERR_UNSUPPORTED otherwise).
 * Counts and offsets stay on the device: the call needs no host synchronisation.
 */
MOE_API int moe_gemm1_swiglu(const void* a, int a_dtype, const uint8_t* a_scale, int layout,
                     const int32_t* expert_counts, const int32_t* expert_offsets,
                     int max_tokens, int64_t rows_cap, int E, int64_t K, int64_t I,
                     const void* w1, const uint8_t* w1_scale, int w_dtype, int w1_layout,
                     int impl, void* h, int h_dtype, uint8_t* h_scale, int32_t* err_word, void* stream);

/*
 * moe_gemm2 -- grouped GEMM with W2 ("Fused MoE Modular Kernel", apply():
 * Matmul with W2), whose epilogue multiplies by the route weight (optional)
 * and writes each result straight to its (token, top-k slot) row ("Cake
 * MegaMoE EP16" FlashInfer PR 5148 analysis, section 3: FC2 results returned
 * directly to the source (token, top-k slot) buffer).
 * For every valid row s of expert e:  y_s[n] = w * sum_i h[s,i] W2[e, n, i],  n < K.
 *
 *   h             (rows, I) of h_dtype (BF16, F32 for the SIMT path, or E4M3 codes), row
 *                 indexing as in moe_gemm1_swiglu
 *   h_scale       E4M3 h ("Fused MoE Modular Kernel", apply(): quantisation between
 *                 act+mul and W2): E8M0 bytes (rows, I/32), 4-byte aligned; NULL otherwise.
 *                 As for GEMM 1, E4M3 h needs E4M3 weights (I % 128 == 0, K % 128 == 0
 *                 on tcgen05 tiles).
 *   w2            (E, K, I) of w_dtype; w2_scale (E, K, I/32) E8M0 for E4M3, else NULL
 *   w2_layout     MOE_W1_GATE_UP (row-major, as above) or MOE_W_TILED (W2 from
 *                 moe_tile_weights, which = 2: bf16 on CTA-pair tiles, E4M3 codes on swap-AB
 *                 tiles, as for moe_gemm1_swiglu)
 *   contiguous:   row s goes to y[row_route[s]] (rows with row_route -1 are skipped);
 *                 y is (y_rows, K) with y_rows = T*top_k; route_weights, if not NULL,
 *                 is (T*top_k) fp32 indexed by route.
 *   batched:      row s goes to y[s]; y is (E*max_tokens, K); route_weights, if not
 *                 NULL, is (E*max_tokens) indexed by row; row_route may be NULL.
 *   y             y_dtype F32 or BF16.
 */
MOE_API int moe_gemm2(const void* h, int h_dtype, const uint8_t* h_scale, int layout,
              const int32_t* expert_counts, const int32_t* expert_offsets,
              int max_tokens, int64_t rows_cap, int E, int64_t K, int64_t I,
              const void* w2, const uint8_t* w2_scale, int w_dtype, int w2_layout,
              const int32_t* row_route, const float* route_weights,
              int impl, void* y, int y_dtype, int64_t y_rows, int32_t* err_word, void* stream);

/*
 * moe_experts_fused -- moe_gemm1_swiglu followed by moe_gemm2 in ONE launch
 * (the "model kernel" of the two-kernel run in the "Cake MegaMoE EP16"
 * FlashInfer PR 5148 analysis, section 4: the experts' GEMMs, then a separate
 * ordered Top-K reduce).  For the decode regime (few tokens per expert):
 * bf16 activations and weights, swap-AB tcgen05 tiles, contiguous layout.
 * GEMM 1 tiles run first; the GEMM 2 tiles of a token segment start once the
 * GEMM 1 tiles of that segment have written their h, so GEMM 2's weights
 * stream while GEMM 1's last tiles finish and no second launch is paid.
 * Results equal moe_gemm1_swiglu + moe_gemm2 with MOE_IMPL_TCGEN05_SWAP_AB.
 *
 *   a, counts, offsets, rows_cap, E, K, I, w1, w1_layout   as moe_gemm1_swiglu
 *   w2, row_route, route_weights, y, y_dtype, y_rows        as moe_gemm2 (contiguous)
 *   a_dtype, w_dtype   MOE_BF16
 *   h          caller-owned (rows_cap, I) BF16 buffer for the intermediate; must not
 *              alias a or y; holds h on return
 *   workspace  >= moe_experts_fused_workspace_size(rows_cap, E) bytes, 256-byte
 *              aligned; cleared by the call (an asynchronous memset on `stream`)
 *   w1_layout  MOE_W1_GATE_UP or MOE_W1_INTERLEAVE16 (W2 row-major), or MOE_W_TILED:
 *              w1 and w2 both as written by moe_tile_weights (same results, bit for bit)
 *   K % 128 == 0, I % 64 == 0; an sm_100+ device.
 * The launch is cooperative (every CTA resident); a wait that runs out sets
 * MOE_DEVERR_TIMEOUT after 2 s instead of hanging.
 */
MOE_API size_t moe_experts_fused_workspace_size(int64_t rows_cap, int E);

/*
 * moe_tile_weights -- offline re-layout of expert weights (bf16, or E4M3 codes) into the
 * tile-contiguous layout that the GEMMs stream with MOE_W_TILED (a
 * weight-preparation step, like the gate/up interleave of the "Cake MegaMoE
 * EP16" FlashInfer PR 5148 analysis, section 2, or the MXFP8 quantisation):
 * every 128-row x 128-byte block that one pipeline stage loads (64 bf16 or 128
 * E4M3 codes per row) is stored as one contiguous 16 KB run, so each stage
 * reads whole DRAM pages instead of 128 pieces of 128 bytes one weight row apart.
 *     out[e][b][c][r][j] = w[e][row(b, r)][n*c + j]
 *     (n = 64 for bf16, 128 for E4M3; b < rows/128, c < cols/n, r < 128, j < n)
 *   which = 1: w is W1 (E, 2I, K) in layout w1_layout; rows = 2I, cols = K; each
 *              block holds 64 gate/up units as [16 gate rows, the 16 matching
 *              up rows] x 4: row(b, r) = unit u = 64b + 16(r/32) + r%16, its gate
 *              row (r%32 < 16) or up row (r%32 >= 16) -- for MOE_W1_GATE_UP
 *              rows u and I + u, for MOE_W1_INTERLEAVE16 row 128b + r.
 *   which = 2: w is W2 (E, K, I); rows = K, cols = I; row(b, r) = 128b + r.
 *   w_dtype    MOE_BF16 (cols % 64 == 0), or MOE_E4M3 codes (cols % 128 == 0; W1
 *              only in MOE_W1_INTERLEAVE16, so that the rows keep their stored order
 *              and the E8M0 scale arrays are used as they are; MOE_ERR_UNSUPPORTED
 *              for [gate; up] codes).  rows % 128 == 0.
 *   w, out     device, 16-byte aligned, E*rows*cols elements each, not overlapping.
 */
MOE_API int moe_tile_weights(const void* w, int w_dtype, int which, int w1_layout, int E, int64_t rows,
                             int64_t cols, void* out, void* stream);
MOE_API int moe_experts_fused(const void* a, int a_dtype, const int32_t* expert_counts,
                              const int32_t* expert_offsets, int64_t rows_cap, int E, int64_t K, int64_t I,
                              const void* w1, int w1_layout, const void* w2, int w_dtype,
                              const int32_t* row_route, const float* route_weights, void* h, void* y,
                              int y_dtype, int64_t y_rows, void* workspace, size_t workspace_bytes,
                              int32_t* err_word, void* stream);

/*
 * moe_unpermute_topk_reduce -- ordered TopK weight-and-reduce
 * ("Fused MoE Modular Kernel", TopKWeightAndReduce, Contiguous; "Cake
 * MegaMoE EP16" analysis, section 4: a separate ordered Top-K reduce kernel).
 *     out[t, n] = sum_{j = 0..top_k-1, 0 <= topk_ids[t,j] < E} w[t,j] * y[t*top_k + j, n]
 * summed in fp32 in increasing j (run-to-run bit-identical); w = 1 when
 * topk_weights is NULL (weights already applied by moe_gemm2).  A token with
 * no valid slot gets +0.0.
 *   y    (T*top_k, K) of y_dtype (F32 or BF16); out (T, K) of out_dtype (F32 or BF16).
 *   K*element size must be a multiple of 16 bytes.
 */
MOE_API int moe_unpermute_topk_reduce(const void* y, int y_dtype, const int32_t* topk_ids, const float* topk_weights,
                              int64_t T, int top_k, int E, int64_t K, void* out, int out_dtype, void* stream);

/*
 * moe_batched_weight_reduce -- naive-batched weight application
 * ("Fused MoE Modular Kernel", TopKWeightAndReduce, NaiveBatched), read as a
 * per-row weight in place of the batched layout:
 *     out[e, q, :] = w[e, q] * y[e, q, :]   for q < expert_num_tokens[e]
 * (w = 1 when row_weights is NULL).  Rows q >= expert_num_tokens[e] are
 * neither read nor written.  y, out: (E, max_tokens, K); out may equal y.
 */
MOE_API int moe_batched_weight_reduce(const void* y, int y_dtype, const int32_t* expert_num_tokens,
                              const float* row_weights, int E, int max_tokens, int64_t K,
                              void* out, int out_dtype, void* stream);

/*
 * moe_batched_topk_reduce -- TopKWeightAndReduce for the Batched format
 * carried through to token order ("Fused MoE Modular Kernel",
 * TopKWeightAndReduce, NaiveBatched; Introduction: the Batched format):
 *     out[t, n] = sum_{j = 0..top_k-1, route_row[t*top_k+j] != -1} w[t,j] * y[route_row[t*top_k+j], n]
 * in increasing j, accumulated in fp32 from +0.0 (a token without a kept route
 * gets +0.0).
 *   y            (rows, K) F32 or BF16 -- for the batched layout the
 *                (E, max_tokens, K) expert outputs, rows = E*max_tokens
 *   route_row    (T*top_k) int32 from moe_permute_align: the row of each
 *                route, -1 for padding and for routes dropped by capacity;
 *                other entries outside [0, rows) set MOE_DEVERR_ID_RANGE in
 *                err_word (may be NULL) and are skipped
 *   topk_weights (T, top_k) fp32 or NULL (weights already applied)
 *   out          (T, K) F32 or BF16, must not alias y
 *   K % 8 == 0; y and out 16-byte aligned.
 * The result does not depend on the launch: the same inputs give the same bits.
 */
MOE_API int moe_batched_topk_reduce(const void* y, int y_dtype, int64_t rows, const int32_t* route_row,
                                    const float* topk_weights, int64_t T, int top_k, int64_t K,
                                    void* out, int out_dtype, int32_t* err_word, void* stream);

/*
 * mxfp8_quantize_block32 -- MXFP8 block-32 quantisation along rows
 * ("Cake MegaMoE EP16" FlashInfer PR 5148 analysis, section 2,
 * _quantize_mxfp8_block32 "After").  For each block of 32 consecutive
 * elements of a row with m = max |x|:
 *     code  = 0 if m == 0, else clamp(ceil(log2(m/448)) + 127, 0, 254)
 *     q[i]  = E4M3(x[i] / 2^(code-127)), round to nearest even, saturating, sign kept.
 *   x       (rows, cols) F32 or BF16; cols % 32 == 0
 *   codes   (rows, cols) uint8 out;  scales (rows, cols/32) uint8 out.
 * The codes and scales are exact (they depend on no rounding order).
 */
MOE_API int mxfp8_quantize_block32(const void* x, int x_dtype, int64_t rows, int64_t cols,
                           uint8_t* codes, uint8_t* scales, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LAYER_H */
