// The C ABI of libmoe_layer: argument validation on the host (nothing is
// launched when a check fails), dispatch to the kernels, error messages.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <mutex>
#include <string>

#include "internal.h"
#include "moe_layer.h"

namespace moe {

namespace {
thread_local std::string g_last_error;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int esize(int dt) { return dt == MOE_F32 ? 4 : (dt == MOE_BF16 ? 2 : 1); }
bool is_float_dtype(int dt) { return dt == MOE_F32 || dt == MOE_BF16; }
cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// T >= 0 and 1 <= top_k <= 1024 with T*top_k < 2^31, tested without forming the product (a huge T would
// overflow it).
bool routes_in_range(int64_t T, int top_k) {
    return T >= 0 && top_k >= 1 && top_k <= 1024 && T <= int64_t(INT32_MAX) / top_k;
}

int launch_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return MOE_OK;
    return fail(MOE_ERR_LAUNCH, std::string(what) + ": " + cudaGetErrorString(e));
}

#define MOE_REQUIRE(cond, status, msg) \
    do {                               \
        if (!(cond)) return fail(status, msg); \
    } while (0)

}  // namespace

int fail(int status, const std::string& msg) {
    g_last_error = msg;
    return status;
}

int check_launch(const char* what) { return launch_status(cudaGetLastError(), what); }

int num_sms() {
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

int device_cc() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return 0;
    return major * 10 + minor;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_last_error(void) { return g_last_error.c_str(); }

int moe_version(void) { return (1 << 16) | 0; }

int64_t moe_max_padded_rows(int64_t T, int top_k, int E, int block_m) {
    if (!routes_in_range(T, top_k) || E < 1 || E > 1024 || block_m < 1 || block_m > 4096) return -1;
    return T * top_k + int64_t(E) * (block_m - 1);
}

size_t moe_permute_workspace_size(int64_t T, int top_k, int E) {
    if (!routes_in_range(T, top_k) || E < 1 || E > 1024) return 0;
    return permute_workspace_bytes(T, top_k, E);
}

int moe_topk_route(const float* logits, int64_t T, int E, int top_k, int renormalize, int32_t* topk_ids,
                   float* topk_weights, void* stream) {
    g_last_error.clear();
    MOE_REQUIRE(T >= 0, MOE_ERR_INVALID_ARG, "moe_topk_route: T < 0");
    MOE_REQUIRE(E >= 1 && E <= 1024, MOE_ERR_INVALID_ARG, "moe_topk_route: E must be in [1, 1024]");
    MOE_REQUIRE(top_k >= 1 && top_k <= std::min(E, 32), MOE_ERR_INVALID_ARG,
                "moe_topk_route: top_k must be in [1, min(E, 32)]");
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(logits && topk_ids && topk_weights, MOE_ERR_INVALID_ARG, "moe_topk_route: null pointer");
    return launch_status(launch_topk_route(logits, T, E, top_k, renormalize, topk_ids, topk_weights,
                                           as_stream(stream)),
                         "moe_topk_route");
}

namespace {

// Argument checks of moe_permute_align (the routing ids are checked by the caller).
int validate_permute(const char* name, int64_t T, int top_k, int E, int layout, int block_m, int max_tokens,
                     const void* x, int x_dtype, int64_t K, const void* x_out, int64_t rows_cap,
                     const int32_t* expert_counts, const int32_t* expert_offsets, const int32_t* row_route,
                     const int32_t* route_row, const void* workspace, size_t workspace_bytes) {
    const std::string n(name);
    MOE_REQUIRE(T >= 0 && top_k >= 1 && top_k <= 1024, MOE_ERR_INVALID_ARG, n + ": bad T or top_k");
    MOE_REQUIRE(routes_in_range(T, top_k), MOE_ERR_INVALID_ARG, n + ": T*top_k must stay below 2^31");
    MOE_REQUIRE(E >= 1 && E <= 1024, MOE_ERR_INVALID_ARG, n + ": E must be in [1, 1024]");
    MOE_REQUIRE(layout == MOE_LAYOUT_CONTIGUOUS || layout == MOE_LAYOUT_BATCHED, MOE_ERR_INVALID_ARG,
                n + ": unknown layout");
    if (layout == MOE_LAYOUT_CONTIGUOUS) {
        MOE_REQUIRE(block_m >= 1 && block_m <= 4096, MOE_ERR_INVALID_ARG, n + ": block_m in [1, 4096]");
        MOE_REQUIRE(rows_cap >= moe_max_padded_rows(T, top_k, E, block_m), MOE_ERR_INVALID_ARG,
                    n + ": rows_cap < T*top_k + E*(block_m-1)");
    } else {
        MOE_REQUIRE(max_tokens >= 0, MOE_ERR_INVALID_ARG, n + ": max_tokens < 0");
        MOE_REQUIRE(rows_cap == int64_t(E) * max_tokens, MOE_ERR_INVALID_ARG,
                    n + ": batched rows_cap must equal E*max_tokens");
    }
    MOE_REQUIRE(rows_cap < (int64_t(1) << 31), MOE_ERR_INVALID_ARG, n + ": rows_cap >= 2^31");
    MOE_REQUIRE(expert_counts && expert_offsets && (row_route || rows_cap == 0) && (route_row || T == 0),
                MOE_ERR_INVALID_ARG, n + ": null output pointer");
    const size_t need = permute_workspace_bytes(T, top_k, E);
    MOE_REQUIRE(workspace_bytes >= need, MOE_ERR_WORKSPACE_TOO_SMALL,
                n + ": workspace smaller than moe_permute_workspace_size()");
    MOE_REQUIRE(workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, MOE_ERR_ALIGNMENT,
                n + ": workspace must be 256-byte aligned");
    if (x) {
        MOE_REQUIRE(is_float_dtype(x_dtype), MOE_ERR_UNSUPPORTED, n + ": x must be F32 or BF16");
        MOE_REQUIRE(K > 0 && (K * esize(x_dtype)) % 16 == 0, MOE_ERR_ALIGNMENT,
                    n + ": K * element size must be a multiple of 16 bytes");
        MOE_REQUIRE(K * esize(x_dtype) < (int64_t(1) << 31), MOE_ERR_INVALID_ARG, n + ": rows of 2^31 bytes or more");
        MOE_REQUIRE(x_out || rows_cap == 0, MOE_ERR_INVALID_ARG, n + ": x given without x_out");
        MOE_REQUIRE(aligned16(x) && aligned16(x_out), MOE_ERR_ALIGNMENT,
                    n + ": x and x_out must be 16-byte aligned");
    }
    return MOE_OK;
}

// The permute launches (and the gather when x is given) of validated arguments.
int run_permute(const char* name, const int32_t* topk_ids, int64_t T, int top_k, int E, int layout, int block_m,
                int max_tokens, const void* x, int x_dtype, int64_t K, void* x_out, int64_t rows_cap,
                int32_t* expert_counts, int32_t* expert_offsets, int32_t* row_route, int32_t* route_row,
                void* workspace, int32_t* err_word, cudaStream_t s) {
    int rc = launch_status(launch_permute(topk_ids, T, top_k, E, layout, block_m, max_tokens, expert_counts,
                                          expert_offsets, row_route, route_row, workspace, err_word, s),
                           name);
    if (rc || !x) return rc;
    return launch_status(launch_gather_rows(x, esize(x_dtype), K, row_route, top_k,
                                            layout == MOE_LAYOUT_CONTIGUOUS ? expert_offsets : nullptr, E,
                                            rows_cap, x_out, s),
                         name);
}

}  // namespace

int moe_permute_align(const int32_t* topk_ids, int64_t T, int top_k, int E, int layout, int block_m,
                      int max_tokens, const void* x, int x_dtype, int64_t K, void* x_out, int64_t rows_cap,
                      int32_t* expert_counts, int32_t* expert_offsets, int32_t* row_route, int32_t* route_row,
                      void* workspace, size_t workspace_bytes, int32_t* err_word, void* stream) {
    g_last_error.clear();
    int rc = validate_permute("moe_permute_align", T, top_k, E, layout, block_m, max_tokens, x, x_dtype, K, x_out,
                              rows_cap, expert_counts, expert_offsets, row_route, route_row, workspace,
                              workspace_bytes);
    if (rc) return rc;
    MOE_REQUIRE(topk_ids || T == 0, MOE_ERR_INVALID_ARG, "moe_permute_align: null topk_ids");
    return run_permute("moe_permute_align", topk_ids, T, top_k, E, layout, block_m, max_tokens, x, x_dtype, K,
                       x_out, rows_cap, expert_counts, expert_offsets, row_route, route_row, workspace, err_word,
                       as_stream(stream));
}

int moe_route_permute_align(const float* logits, int64_t T, int E, int top_k, int renormalize, int32_t* topk_ids,
                            float* topk_weights, int layout, int block_m, int max_tokens, const void* x,
                            int x_dtype, int64_t K, void* x_out, int64_t rows_cap, int32_t* expert_counts,
                            int32_t* expert_offsets, int32_t* row_route, int32_t* route_row, void* workspace,
                            size_t workspace_bytes, int32_t* err_word, void* stream) {
    g_last_error.clear();
    const char* name = "moe_route_permute_align";
    MOE_REQUIRE(top_k >= 1 && top_k <= std::min(E, 32), MOE_ERR_INVALID_ARG,
                "moe_route_permute_align: top_k must be in [1, min(E, 32)]");
    int rc = validate_permute(name, T, top_k, E, layout, block_m, max_tokens, x, x_dtype, K, x_out, rows_cap,
                              expert_counts, expert_offsets, row_route, route_row, workspace, workspace_bytes);
    if (rc) return rc;
    MOE_REQUIRE((logits && topk_ids && topk_weights) || T == 0, MOE_ERR_INVALID_ARG,
                "moe_route_permute_align: null logits, topk_ids or topk_weights");
    cudaStream_t s = as_stream(stream);
    const int64_t row_bytes = x ? K * esize(x_dtype) : 0;
    if (route_permute_fusable(T, top_k, row_bytes))
        return launch_status(launch_route_permute(logits, T, E, top_k, renormalize, topk_ids, topk_weights, layout,
                                                  block_m, max_tokens, expert_counts, expert_offsets, row_route,
                                                  route_row, x, row_bytes, x ? x_out : nullptr, err_word, s),
                             name);
    if (T > 0) {
        rc = launch_status(launch_topk_route(logits, T, E, top_k, renormalize, topk_ids, topk_weights, s), name);
        if (rc) return rc;
    }
    return run_permute(name, topk_ids, T, top_k, E, layout, block_m, max_tokens, x, x_dtype, K, x_out, rows_cap,
                       expert_counts, expert_offsets, row_route, route_row, workspace, err_word, s);
}

namespace {

int validate_gemm(const GemmArgs& g, const char* name) {
    const std::string n(name);
    MOE_REQUIRE(g.E >= 1 && g.E <= 1024, MOE_ERR_INVALID_ARG, n + ": E must be in [1, 1024]");
    MOE_REQUIRE(g.K > 0 && g.I > 0, MOE_ERR_INVALID_ARG, n + ": K and I must be positive");
    MOE_REQUIRE(g.K % 32 == 0 && g.I % 32 == 0, MOE_ERR_ALIGNMENT, n + ": K and I must be multiples of 32");
    MOE_REQUIRE(g.layout == MOE_LAYOUT_CONTIGUOUS || g.layout == MOE_LAYOUT_BATCHED, MOE_ERR_INVALID_ARG,
                n + ": unknown layout");
    // no rows (an empty batch): the activation and output buffers may be empty (NULL)
    const int64_t rows = g.layout == MOE_LAYOUT_CONTIGUOUS ? g.rows_cap : int64_t(g.E) * g.max_tokens;
    MOE_REQUIRE(g.w && g.counts && ((g.a && g.out) || rows == 0), MOE_ERR_INVALID_ARG, n + ": null pointer");
    MOE_REQUIRE(aligned16(g.a) && aligned16(g.w) && aligned16(g.out), MOE_ERR_ALIGNMENT,
                n + ": activation, weight and output pointers must be 16-byte aligned");
    MOE_REQUIRE((is_float_dtype(g.a_dtype) || g.a_dtype == MOE_E4M3) &&
                    (is_float_dtype(g.out_dtype) || (g.gemm == 1 && g.out_dtype == MOE_E4M3)),
                MOE_ERR_UNSUPPORTED, n + ": activations must be F32, BF16 or E4M3; outputs F32 or BF16 (or E4M3 h)");
    if (g.out_dtype == MOE_E4M3) {
        MOE_REQUIRE(g.out_scale, MOE_ERR_INVALID_ARG, n + ": E4M3 h needs an h_scale output");
        MOE_REQUIRE(g.I % 32 == 0, MOE_ERR_ALIGNMENT, n + ": E4M3 h needs I % 32 == 0");
    }
    if (g.a_dtype == MOE_E4M3) {
        MOE_REQUIRE(g.a_scale, MOE_ERR_INVALID_ARG, n + ": E4M3 activations need scales");
        MOE_REQUIRE((reinterpret_cast<uintptr_t>(g.a_scale) & 3u) == 0, MOE_ERR_ALIGNMENT,
                    n + ": activation scales must be 4-byte aligned");
        MOE_REQUIRE(g.w_dtype == MOE_E4M3, MOE_ERR_UNSUPPORTED, n + ": E4M3 activations need E4M3 weights");
    }
    MOE_REQUIRE(g.w_dtype == MOE_F32 || g.w_dtype == MOE_BF16 || g.w_dtype == MOE_E4M3, MOE_ERR_UNSUPPORTED,
                n + ": unknown weight dtype");
    MOE_REQUIRE(g.w_dtype != MOE_E4M3 || g.w_scale, MOE_ERR_INVALID_ARG, n + ": E4M3 weights need scales");
    if (g.layout == MOE_LAYOUT_CONTIGUOUS) {
        MOE_REQUIRE(g.offsets, MOE_ERR_INVALID_ARG, n + ": contiguous layout needs expert_offsets");
        MOE_REQUIRE(g.rows_cap >= 0 && g.rows_cap < (int64_t(1) << 31), MOE_ERR_INVALID_ARG,
                    n + ": rows_cap out of range");
    } else {
        MOE_REQUIRE(g.max_tokens >= 0, MOE_ERR_INVALID_ARG, n + ": max_tokens < 0");
        MOE_REQUIRE(int64_t(g.E) * g.max_tokens < (int64_t(1) << 31), MOE_ERR_INVALID_ARG,
                    n + ": E*max_tokens >= 2^31");
    }
    return MOE_OK;
}

// E4M3 activations (with E4M3 weights): block-scaled tcgen05 swap-AB tiles, or the CUDA-core kernel.
int run_gemm_mx(const GemmArgs& g, int impl, cudaStream_t s, const char* name) {
    if (impl == MOE_IMPL_SIMT) return launch_status(launch_gemm_simt(g, s), name);
    MOE_REQUIRE(impl == MOE_IMPL_AUTO || impl == MOE_IMPL_TCGEN05_SWAP_AB, MOE_ERR_UNSUPPORTED,
                std::string(name) + ": E4M3 activations run on swap-AB tcgen05 tiles (or SIMT)");
    if (device_cc() < 100) {
        if (impl == MOE_IMPL_AUTO) return launch_status(launch_gemm_simt(g, s), name);
        return fail(MOE_ERR_UNSUPPORTED, std::string(name) + ": tcgen05 needs an sm_100+ device");
    }
    int rc = launch_gemm_mx(g, s);
    if (rc != MOE_OK && impl == MOE_IMPL_AUTO && rc == MOE_ERR_UNSUPPORTED) {
        g_last_error.clear();
        return launch_status(launch_gemm_simt(g, s), name);
    }
    return rc;
}

int run_gemm(const GemmArgs& g, int impl, cudaStream_t s, const char* name) {
    if ((g.layout == MOE_LAYOUT_CONTIGUOUS ? g.rows_cap : int64_t(g.E) * g.max_tokens) == 0) return MOE_OK;
    if (g.w1_layout == MOE_W_TILED && g.w_dtype == MOE_E4M3) {
        // tile-contiguous E4M3 codes are read by the swap-AB tiles: bf16 activations decode them into TMEM, E4M3
        // activations take the block-scaled MMA
        MOE_REQUIRE(impl == MOE_IMPL_AUTO || impl == MOE_IMPL_TCGEN05_SWAP_AB, MOE_ERR_UNSUPPORTED,
                    std::string(name) + ": tile-contiguous E4M3 codes run on swap-AB tiles (MOE_IMPL_TCGEN05_SWAP_AB)");
        MOE_REQUIRE(g.a_dtype == MOE_BF16 || g.a_dtype == MOE_E4M3, MOE_ERR_UNSUPPORTED,
                    std::string(name) + ": tile-contiguous E4M3 codes need bf16 or E4M3 activations");
        MOE_REQUIRE(device_cc() >= 100, MOE_ERR_UNSUPPORTED, std::string(name) + ": tcgen05 needs an sm_100+ device");
        return g.a_dtype == MOE_E4M3 ? launch_gemm_mx(g, s) : launch_gemm_tc(g, TC_SWAP, s);
    }
    if (g.w1_layout == MOE_W_TILED) {
        // tile-contiguous bf16 weights (moe_tile_weights) are read by the CTA-pair tiles
        MOE_REQUIRE(impl == MOE_IMPL_AUTO || impl == MOE_IMPL_TCGEN05_PAIR, MOE_ERR_UNSUPPORTED,
                    std::string(name) + ": tile-contiguous weights run on CTA-pair tiles (MOE_IMPL_TCGEN05_PAIR) only");
        MOE_REQUIRE(g.a_dtype == MOE_BF16 && g.w_dtype == MOE_BF16, MOE_ERR_UNSUPPORTED,
                    std::string(name) + ": tile-contiguous weights need bf16 activations and weights");
        MOE_REQUIRE(device_cc() >= 100, MOE_ERR_UNSUPPORTED, std::string(name) + ": tcgen05 needs an sm_100+ device");
        return launch_gemm_pair(g, s);
    }
    if (g.a_dtype == MOE_E4M3) return run_gemm_mx(g, impl, s, name);
    const bool tc_ok = g.a_dtype == MOE_BF16 && (g.w_dtype == MOE_BF16 || g.w_dtype == MOE_E4M3) &&
                       g.out_dtype == MOE_BF16 && device_cc() >= 100;
    int chosen = impl;
    if (impl == MOE_IMPL_AUTO) {
        if (!tc_ok) {
            chosen = MOE_IMPL_SIMT;
        } else if (g.w_dtype == MOE_E4M3) {
            chosen = MOE_IMPL_TCGEN05_SWAP_AB;     // E4M3 weights are decoded on swap-AB tiles
        } else {
            // few routes per expert (decode): weight rows on the MMA M side
            int64_t rows = g.layout == MOE_LAYOUT_CONTIGUOUS ? g.rows_cap : int64_t(g.E) * g.max_tokens;
            int64_t per_expert = rows / std::max(1, g.E);
            if (g.layout == MOE_LAYOUT_BATCHED) per_expert = g.max_tokens / 2;
            // many tokens per expert: CTA-pair tiles (measured faster than 128-row normal tiles on the skewed
            // prefill, batched and batched-token workloads), normal tiles for shapes outside them
            chosen = per_expert < 64 ? MOE_IMPL_TCGEN05_SWAP_AB
                                     : (g.w_dtype == MOE_BF16 ? MOE_IMPL_TCGEN05_PAIR : MOE_IMPL_TCGEN05);
        }
    }
    if (chosen == MOE_IMPL_SIMT) return launch_status(launch_gemm_simt(g, s), name);
    if (chosen == MOE_IMPL_TCGEN05_PAIR) {
        MOE_REQUIRE(device_cc() >= 100, MOE_ERR_UNSUPPORTED, std::string(name) + ": tcgen05 needs an sm_100+ device");
        const int rc = launch_gemm_pair(g, s);
        if (rc != MOE_ERR_UNSUPPORTED || impl != MOE_IMPL_AUTO) return rc;
        g_last_error.clear();   // shape outside the pair tiles: single-SM normal tiles (or CUDA cores) below
        chosen = MOE_IMPL_TCGEN05;
    }
    MOE_REQUIRE(chosen == MOE_IMPL_TCGEN05 || chosen == MOE_IMPL_TCGEN05_SWAP_AB ||
                    chosen == MOE_IMPL_TCGEN05_MIXED,
                MOE_ERR_INVALID_ARG, std::string(name) + ": unknown impl");
    MOE_REQUIRE(device_cc() >= 100, MOE_ERR_UNSUPPORTED, std::string(name) + ": tcgen05 needs an sm_100+ device");
    const int mode = chosen == MOE_IMPL_TCGEN05_SWAP_AB ? TC_SWAP : (chosen == MOE_IMPL_TCGEN05_MIXED ? TC_MIXED
                                                                                                      : TC_NORMAL);
    int rc = launch_gemm_tc(g, mode, s);
    if (rc != MOE_OK && impl == MOE_IMPL_AUTO && rc == MOE_ERR_UNSUPPORTED) {
        // shape outside the tcgen05 tiles: the CUDA-core kernel covers every shape
        g_last_error.clear();
        return launch_status(launch_gemm_simt(g, s), name);
    }
    return rc;
}

}  // namespace

int moe_gemm1_swiglu(const void* a, int a_dtype, const uint8_t* a_scale, int layout, const int32_t* expert_counts,
                     const int32_t* expert_offsets, int max_tokens, int64_t rows_cap, int E, int64_t K, int64_t I,
                     const void* w1, const uint8_t* w1_scale, int w_dtype, int w1_layout, int impl, void* h,
                     int h_dtype, uint8_t* h_scale, int32_t* err_word, void* stream) {
    g_last_error.clear();
    GemmArgs g{};
    g.gemm = 1;
    g.out_scale = h_scale;
    g.a = a;
    g.a_dtype = a_dtype;
    g.a_scale = a_scale;
    g.layout = layout;
    g.counts = expert_counts;
    g.offsets = layout == MOE_LAYOUT_CONTIGUOUS ? expert_offsets : nullptr;
    g.max_tokens = max_tokens;
    g.rows_cap = layout == MOE_LAYOUT_CONTIGUOUS ? rows_cap : int64_t(E) * max_tokens;
    g.E = E;
    g.K = K;
    g.I = I;
    g.w = w1;
    g.w_scale = w1_scale;
    g.w_dtype = w_dtype;
    g.w1_layout = w1_layout;
    g.out = h;
    g.out_dtype = h_dtype;
    g.err_word = err_word;
    int rc = validate_gemm(g, "moe_gemm1_swiglu");
    if (rc) return rc;
    MOE_REQUIRE(w1_layout == MOE_W1_GATE_UP || w1_layout == MOE_W1_INTERLEAVE16 || w1_layout == MOE_W_TILED,
                MOE_ERR_INVALID_ARG, "moe_gemm1_swiglu: unknown w1_layout");
    MOE_REQUIRE(w1_layout != MOE_W1_INTERLEAVE16 || I % 16 == 0, MOE_ERR_ALIGNMENT,
                "moe_gemm1_swiglu: interleave-16 needs I % 16 == 0");
    return run_gemm(g, impl, as_stream(stream), "moe_gemm1_swiglu");
}

int moe_gemm2(const void* hh, int h_dtype, const uint8_t* h_scale, int layout, const int32_t* expert_counts,
              const int32_t* expert_offsets, int max_tokens, int64_t rows_cap, int E, int64_t K, int64_t I,
              const void* w2, const uint8_t* w2_scale, int w_dtype, int w2_layout, const int32_t* row_route,
              const float* route_weights, int impl, void* y, int y_dtype, int64_t y_rows, int32_t* err_word,
              void* stream) {
    g_last_error.clear();
    GemmArgs g{};
    g.gemm = 2;
    g.a = hh;
    g.a_dtype = h_dtype;
    g.a_scale = h_scale;
    g.layout = layout;
    g.counts = expert_counts;
    g.offsets = layout == MOE_LAYOUT_CONTIGUOUS ? expert_offsets : nullptr;
    g.max_tokens = max_tokens;
    g.rows_cap = layout == MOE_LAYOUT_CONTIGUOUS ? rows_cap : int64_t(E) * max_tokens;
    g.E = E;
    g.K = K;
    g.I = I;
    g.w = w2;
    g.w_scale = w2_scale;
    g.w_dtype = w_dtype;
    g.w1_layout = w2_layout;   // MOE_W1_GATE_UP (row-major) or MOE_W_TILED
    g.row_route = row_route;
    g.route_w = route_weights;
    g.out = y;
    g.out_dtype = y_dtype;
    g.out_rows = y_rows;
    g.err_word = err_word;
    int rc = validate_gemm(g, "moe_gemm2");
    if (rc) return rc;
    MOE_REQUIRE(layout == MOE_LAYOUT_BATCHED || row_route, MOE_ERR_INVALID_ARG,
                "moe_gemm2: contiguous layout needs row_route");
    MOE_REQUIRE(w2_layout == MOE_W1_GATE_UP || w2_layout == MOE_W_TILED, MOE_ERR_INVALID_ARG,
                "moe_gemm2: w2_layout must be MOE_W1_GATE_UP (row-major) or MOE_W_TILED");
    MOE_REQUIRE(y_rows >= 0, MOE_ERR_INVALID_ARG, "moe_gemm2: y_rows < 0");
    return run_gemm(g, impl, as_stream(stream), "moe_gemm2");
}

size_t moe_experts_fused_workspace_size(int64_t rows_cap, int E) {
    if (rows_cap < 0 || E < 1) return 0;
    return experts_fused_workspace_bytes(rows_cap, E);
}

int moe_experts_fused(const void* a, int a_dtype, const int32_t* expert_counts, const int32_t* expert_offsets,
                      int64_t rows_cap, int E, int64_t K, int64_t I, const void* w1, int w1_layout, const void* w2,
                      int w_dtype, const int32_t* row_route, const float* route_weights, void* h, void* y,
                      int y_dtype, int64_t y_rows, void* workspace, size_t workspace_bytes, int32_t* err_word,
                      void* stream) {
    g_last_error.clear();
    GemmArgs g1{};
    g1.gemm = 1;
    g1.a = a;
    g1.a_dtype = a_dtype;
    g1.layout = MOE_LAYOUT_CONTIGUOUS;
    g1.counts = expert_counts;
    g1.offsets = expert_offsets;
    g1.rows_cap = rows_cap;
    g1.E = E;
    g1.K = K;
    g1.I = I;
    g1.w = w1;
    g1.w_dtype = w_dtype;
    g1.w1_layout = w1_layout;
    g1.out = h;
    g1.out_dtype = MOE_BF16;
    g1.err_word = err_word;
    int rc = validate_gemm(g1, "moe_experts_fused");
    if (rc) return rc;
    GemmArgs g2 = g1;
    g2.gemm = 2;
    g2.a = h;
    g2.w = w2;
    g2.w1_layout = w1_layout == MOE_W_TILED ? MOE_W_TILED : 0;   // tiled: W2 tiled as well
    g2.row_route = row_route;
    g2.route_w = route_weights;
    g2.out = y;
    g2.out_dtype = y_dtype;
    g2.out_rows = y_rows;
    rc = validate_gemm(g2, "moe_experts_fused");
    if (rc) return rc;
    MOE_REQUIRE(w1_layout == MOE_W1_GATE_UP || w1_layout == MOE_W1_INTERLEAVE16 || w1_layout == MOE_W_TILED,
                MOE_ERR_INVALID_ARG, "moe_experts_fused: unknown w1_layout");
    MOE_REQUIRE(row_route, MOE_ERR_INVALID_ARG, "moe_experts_fused: row_route is required");
    MOE_REQUIRE(y_rows >= 0, MOE_ERR_INVALID_ARG, "moe_experts_fused: y_rows < 0");
    MOE_REQUIRE(rows_cap == 0 || (h != a && h != y), MOE_ERR_INVALID_ARG,
                "moe_experts_fused: h must not alias a or y");
    MOE_REQUIRE(workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, MOE_ERR_ALIGNMENT,
                "moe_experts_fused: workspace must be 256-byte aligned");
    MOE_REQUIRE(device_cc() >= 100, MOE_ERR_UNSUPPORTED, "moe_experts_fused: tcgen05 needs an sm_100+ device");
    return launch_experts_fused(g1, g2, static_cast<int32_t*>(workspace), workspace_bytes, as_stream(stream));
}

int moe_tile_weights(const void* w, int w_dtype, int which, int w1_layout, int E, int64_t rows, int64_t cols,
                     void* out, void* stream) {
    g_last_error.clear();
    MOE_REQUIRE(w_dtype == MOE_BF16 || w_dtype == MOE_E4M3, MOE_ERR_UNSUPPORTED,
                "moe_tile_weights: bf16 weights or E4M3 codes only");
    MOE_REQUIRE(which == 1 || which == 2, MOE_ERR_INVALID_ARG, "moe_tile_weights: which must be 1 (W1) or 2 (W2)");
    MOE_REQUIRE(which == 2 || w1_layout == MOE_W1_GATE_UP || w1_layout == MOE_W1_INTERLEAVE16, MOE_ERR_INVALID_ARG,
                "moe_tile_weights: unknown w1_layout");
    const bool codes = w_dtype == MOE_E4M3;   // 1-byte elements: a 128 x 128-code block is 16 KB
    MOE_REQUIRE(!codes || which == 2 || w1_layout == MOE_W1_INTERLEAVE16, MOE_ERR_UNSUPPORTED,
                "moe_tile_weights: E4M3 W1 codes must be in the interleave-16 layout (their E8M0 scales keep the "
                "stored row order)");
    MOE_REQUIRE(E >= 1 && rows > 0 && cols > 0, MOE_ERR_INVALID_ARG, "moe_tile_weights: bad sizes");
    MOE_REQUIRE(rows % 128 == 0 && cols % (codes ? 128 : 64) == 0, MOE_ERR_ALIGNMENT,
                codes ? "moe_tile_weights: rows % 128 and cols % 128 must be 0"
                      : "moe_tile_weights: rows % 128 and cols % 64 must be 0");
    MOE_REQUIRE(w && out, MOE_ERR_INVALID_ARG, "moe_tile_weights: null pointer");
    MOE_REQUIRE(aligned16(w) && aligned16(out), MOE_ERR_ALIGNMENT, "moe_tile_weights: w and out must be 16-byte aligned");
    const int64_t bytes = int64_t(E) * rows * cols * (codes ? 1 : 2);
    const uintptr_t a = reinterpret_cast<uintptr_t>(w), b = reinterpret_cast<uintptr_t>(out);
    MOE_REQUIRE(a + uintptr_t(bytes) <= b || b + uintptr_t(bytes) <= a, MOE_ERR_INVALID_ARG,
                "moe_tile_weights: w and out overlap");
    // E4M3 codes move as pairs: the same 128-byte row pieces as 64 bf16 columns
    return launch_status(launch_tile_weights(w, which, w1_layout, E, rows, codes ? cols / 2 : cols, out,
                                             as_stream(stream)),
                         "moe_tile_weights");
}

int moe_unpermute_topk_reduce(const void* y, int y_dtype, const int32_t* topk_ids, const float* topk_weights,
                              int64_t T, int top_k, int E, int64_t K, void* out, int out_dtype, void* stream) {
    g_last_error.clear();
    MOE_REQUIRE(routes_in_range(T, top_k) && E >= 1 && K > 0, MOE_ERR_INVALID_ARG,
                "moe_unpermute_topk_reduce: bad sizes (T*top_k must stay below 2^31)");
    MOE_REQUIRE(is_float_dtype(y_dtype) && is_float_dtype(out_dtype), MOE_ERR_UNSUPPORTED,
                "moe_unpermute_topk_reduce: y and out must be F32 or BF16");
    MOE_REQUIRE(K % 8 == 0, MOE_ERR_ALIGNMENT, "moe_unpermute_topk_reduce: K must be a multiple of 8");
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(y && topk_ids && out, MOE_ERR_INVALID_ARG, "moe_unpermute_topk_reduce: null pointer");
    MOE_REQUIRE(aligned16(y) && aligned16(out), MOE_ERR_ALIGNMENT,
                "moe_unpermute_topk_reduce: y and out must be 16-byte aligned");
    return launch_status(launch_topk_reduce(y, y_dtype, topk_ids, topk_weights, T, top_k, E, K, out, out_dtype,
                                            as_stream(stream)),
                         "moe_unpermute_topk_reduce");
}

int moe_batched_weight_reduce(const void* y, int y_dtype, const int32_t* expert_num_tokens,
                              const float* row_weights, int E, int max_tokens, int64_t K, void* out, int out_dtype,
                              void* stream) {
    g_last_error.clear();
    MOE_REQUIRE(E >= 1 && max_tokens >= 0 && K > 0, MOE_ERR_INVALID_ARG, "moe_batched_weight_reduce: bad sizes");
    MOE_REQUIRE(int64_t(E) * max_tokens < (int64_t(1) << 31), MOE_ERR_INVALID_ARG,
                "moe_batched_weight_reduce: E * max_tokens must be below 2^31");
    MOE_REQUIRE(is_float_dtype(y_dtype) && is_float_dtype(out_dtype), MOE_ERR_UNSUPPORTED,
                "moe_batched_weight_reduce: y and out must be F32 or BF16");
    MOE_REQUIRE(K % 8 == 0, MOE_ERR_ALIGNMENT, "moe_batched_weight_reduce: K must be a multiple of 8");
    MOE_REQUIRE(y && expert_num_tokens && out, MOE_ERR_INVALID_ARG, "moe_batched_weight_reduce: null pointer");
    MOE_REQUIRE(aligned16(y) && aligned16(out), MOE_ERR_ALIGNMENT,
                "moe_batched_weight_reduce: y and out must be 16-byte aligned");
    if (y == out && esize(y_dtype) != esize(out_dtype))
        return fail(MOE_ERR_INVALID_ARG, "moe_batched_weight_reduce: in place needs the same element type");
    return launch_status(launch_batched_weight(y, y_dtype, expert_num_tokens, row_weights, E, max_tokens, K, out,
                                               out_dtype, as_stream(stream)),
                         "moe_batched_weight_reduce");
}

int moe_batched_topk_reduce(const void* y, int y_dtype, int64_t rows, const int32_t* route_row,
                            const float* topk_weights, int64_t T, int top_k, int64_t K, void* out, int out_dtype,
                            int32_t* err_word, void* stream) {
    g_last_error.clear();
    MOE_REQUIRE(routes_in_range(T, top_k) && rows >= 0 && K > 0, MOE_ERR_INVALID_ARG,
                "moe_batched_topk_reduce: bad sizes (T*top_k must stay below 2^31)");
    MOE_REQUIRE(rows <= INT32_MAX, MOE_ERR_INVALID_ARG, "moe_batched_topk_reduce: rows must fit int32");
    MOE_REQUIRE(is_float_dtype(y_dtype) && is_float_dtype(out_dtype), MOE_ERR_UNSUPPORTED,
                "moe_batched_topk_reduce: y and out must be F32 or BF16");
    MOE_REQUIRE(K % 8 == 0, MOE_ERR_ALIGNMENT, "moe_batched_topk_reduce: K must be a multiple of 8");
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(route_row && out && (y || rows == 0), MOE_ERR_INVALID_ARG, "moe_batched_topk_reduce: null pointer");
    MOE_REQUIRE(y != out, MOE_ERR_INVALID_ARG, "moe_batched_topk_reduce: out must not alias y");
    MOE_REQUIRE((!y || aligned16(y)) && aligned16(out), MOE_ERR_ALIGNMENT,
                "moe_batched_topk_reduce: y and out must be 16-byte aligned");
    return launch_status(launch_rows_topk_reduce(y, y_dtype, rows, route_row, topk_weights, T, top_k, K, out,
                                                 out_dtype, err_word, as_stream(stream)),
                         "moe_batched_topk_reduce");
}

int mxfp8_quantize_block32(const void* x, int x_dtype, int64_t rows, int64_t cols, uint8_t* codes,
                           uint8_t* scales, void* stream) {
    g_last_error.clear();
    MOE_REQUIRE(rows >= 0 && cols >= 0, MOE_ERR_INVALID_ARG, "mxfp8_quantize_block32: negative size");
    MOE_REQUIRE(cols % 32 == 0, MOE_ERR_ALIGNMENT, "mxfp8_quantize_block32: cols must be a multiple of 32");
    MOE_REQUIRE(is_float_dtype(x_dtype), MOE_ERR_UNSUPPORTED, "mxfp8_quantize_block32: x must be F32 or BF16");
    if (rows == 0 || cols == 0) return MOE_OK;
    MOE_REQUIRE(x && codes && scales, MOE_ERR_INVALID_ARG, "mxfp8_quantize_block32: null pointer");
    MOE_REQUIRE(aligned16(x) && aligned16(codes), MOE_ERR_ALIGNMENT,
                "mxfp8_quantize_block32: x and codes must be 16-byte aligned");
    return launch_status(launch_mxfp8_quantize(x, x_dtype, rows, cols, codes, scales, as_stream(stream)),
                         "mxfp8_quantize_block32");
}

}  // extern "C"
