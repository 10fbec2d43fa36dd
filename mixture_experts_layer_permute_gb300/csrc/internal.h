// Host-side launchers shared between the translation units of libmoe_layer.
// Arguments are validated in api.cu before any of these is called.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>

namespace moe {

// Records a message for moe_last_error() and returns `status`.
int fail(int status, const std::string& msg);
// Checks cudaGetLastError() after a launch; returns MOE_OK or MOE_ERR_LAUNCH.
int check_launch(const char* what);

int num_sms();
int device_cc();   // major*10 + minor of the current device, 0 if none

cudaError_t launch_topk_route(const float* logits, int64_t T, int E, int top_k, int renorm, int32_t* ids,
                              float* weights, cudaStream_t s);

size_t permute_workspace_bytes(int64_t T, int top_k, int E);
cudaError_t launch_permute(const int32_t* ids, int64_t T, int top_k, int E, int layout, int block_m,
                           int max_tokens, int32_t* counts, int32_t* offsets, int32_t* row_route,
                           int32_t* route_row, void* ws, int32_t* err_word, cudaStream_t s);
cudaError_t launch_gather_rows(const void* x, int esize, int64_t K, const int32_t* row_route, int top_k,
                               const int32_t* offsets, int E, int64_t rows_cap, void* x_out, cudaStream_t s);

// tile-contiguous weight layout (moe_tile_weights)
cudaError_t launch_tile_weights(const void* w, int which, int w1_layout, int E, int64_t rows, int64_t cols,
                                void* out, cudaStream_t s);

// route + permute (+ gather when x_out is set) in one launch; only for the sizes route_permute_fusable accepts
bool route_permute_fusable(int64_t T, int top_k, int64_t row_bytes);
cudaError_t launch_route_permute(const float* logits, int64_t T, int E, int top_k, int renorm, int32_t* ids,
                                 float* weights, int layout, int block_m, int max_tokens, int32_t* counts,
                                 int32_t* offsets, int32_t* row_route, int32_t* route_row, const void* x,
                                 int64_t row_bytes, void* x_out, int32_t* err_word, cudaStream_t s);

cudaError_t launch_topk_reduce(const void* y, int y_dtype, const int32_t* ids, const float* w, int64_t T,
                               int top_k, int E, int64_t K, void* out, int out_dtype, cudaStream_t s);
cudaError_t launch_rows_topk_reduce(const void* y, int y_dtype, int64_t rows, const int32_t* route_row,
                                    const float* w, int64_t T, int top_k, int64_t K, void* out, int out_dtype,
                                    int32_t* err_word, cudaStream_t s);
cudaError_t launch_batched_weight(const void* y, int y_dtype, const int32_t* counts, const float* w, int E,
                                  int max_tokens, int64_t K, void* out, int out_dtype, cudaStream_t s);

cudaError_t launch_mxfp8_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, uint8_t* codes,
                                  uint8_t* scales, cudaStream_t s);

struct GemmArgs {
    int gemm;               // 1: gate/up + SiLU-and-mul, 2: down projection
    const void* a;          // activations (gemm 1) or h (gemm 2)
    int a_dtype;
    const uint8_t* a_scale; // E4M3 activations: E8M0 scales (rows, kdim/32)
    int layout;
    const int32_t* counts;
    const int32_t* offsets; // contiguous layout; NULL for batched
    int max_tokens;
    int64_t rows_cap;
    int E;
    int64_t K, I;
    const void* w;
    const uint8_t* w_scale;
    int w_dtype;
    int w1_layout;
    const int32_t* row_route;   // gemm 2, contiguous
    const float* route_w;       // gemm 2, optional
    void* out;
    int out_dtype;
    uint8_t* out_scale;     // GEMM 1 with E4M3 h: E8M0 scales of h (rows, I/32)
    int64_t out_rows;
    int32_t* err_word;
};

cudaError_t launch_gemm_simt(const GemmArgs& g, cudaStream_t s);
// tcgen05 tile kinds: tokens on the MMA M side, weights on M (swap-AB), or both in one launch.
enum { TC_NORMAL = 0, TC_SWAP = 1, TC_MIXED = 2 };
// Returns MOE_OK or a status (with message) when the tcgen05 path cannot run.
int launch_gemm_tc(const GemmArgs& g, int mode, cudaStream_t s);
// TMA tensor maps of one tcgen05 launch: activation rows and weight rows (normal or swap-AB boxes), and for
// mixed launches the swap-AB pair as well; encoded once per (device, pointers, shape) and cached.
struct MapSet {
    CUtensorMap act, w, act_s, w_s;
};
int cached_maps(const GemmArgs& g, int mode, bool w8, int64_t kdim, int64_t wrows, int w_mode, MapSet* out);
// bf16 grouped GEMM on CTA pairs (cta_group::2): 256 weight rows across the two SMs of a pair, up to 256 tokens
// per tile.  Returns MOE_ERR_UNSUPPORTED (nothing launched) for shapes outside its tiles.
int launch_gemm_pair(const GemmArgs& g, cudaStream_t s);
// GEMM 1 then GEMM 2 (bf16, swap-AB tiles, contiguous layout) in one cooperative launch; seg_done is the
// caller's workspace (per token segment counters, cleared by the call).
size_t experts_fused_workspace_bytes(int64_t rows_cap, int E);
int launch_experts_fused(const GemmArgs& g1, const GemmArgs& g2, int32_t* seg_done, size_t ws_bytes,
                         cudaStream_t s);
// Test hook of the bounded waits (MOE_TEST_SKIP_FIRST_COPY=1 at the first launch): CTA 0 of each tcgen05 GEMM
// announces its first stage's bytes but never issues the copy.
bool timeout_test_hook();
// Block-scaled MXFP8 (E4M3 activations and weights) on swap-AB tcgen05 tiles.
int launch_gemm_mx(const GemmArgs& g, cudaStream_t s);

}  // namespace moe
