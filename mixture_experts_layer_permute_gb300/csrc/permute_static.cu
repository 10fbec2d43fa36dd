// moe_permute_align_static: moe_permute_align for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand us a workspace: code running inside a host
// framework that owns every byte of device memory and gives plugins no
// allocator, services that forbid cudaMalloc/cudaFree on their request path
// (both can synchronise the whole device and stall other streams), or
// embedded deployments whose memory budget is fixed at start-up.  For them
// this entry point keeps its scratch in a fixed array that lives in the
// library's own device image instead of in caller-provided memory.
//
// The array below is reserved on every GPU that loads this library and is
// held until the process exits.  Its device address is looked up once per
// device with cudaGetSymbolAddress (the first call on a device does that
// look-up, so make that first call before any stream capture).  All calls
// share the one array, so two calls that overlap on the GPU (different
// streams, or different host threads on one device) race on it and must be
// serialised by the caller.  Nothing in the scratch has to start at zero:
// each call writes every entry it later reads.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "internal.h"
#include "moe_layer.h"

namespace moe {

namespace {

constexpr size_t kStaticScratchBytes = size_t(2) << 20;   // 2 MiB

static __device__ __align__(256) unsigned char g_permute_scratch[kStaticScratchBytes];

// Device address of g_permute_scratch on the current device (looked up once per device).
int static_scratch(void** out) {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(MOE_ERR_LAUNCH, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(MOE_ERR_UNSUPPORTED, "moe_permute_align_static: device index >= 64");
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_permute_scratch);
        if (e != cudaSuccess || !p)
            return fail(MOE_ERR_LAUNCH,
                        std::string("cudaGetSymbolAddress(g_permute_scratch): ") + cudaGetErrorString(e));
        addr[dev] = p;
    }
    *out = addr[dev];
    return MOE_OK;
}

}  // namespace

}  // namespace moe

extern "C" MOE_API int moe_permute_align_static(const int32_t* topk_ids, int64_t T, int top_k, int E, int layout,
                                                int block_m, int max_tokens, const void* x, int x_dtype, int64_t K,
                                                void* x_out, int64_t rows_cap, int32_t* expert_counts,
                                                int32_t* expert_offsets, int32_t* row_route, int32_t* route_row,
                                                int32_t* err_word, void* stream) {
    using namespace moe;
    if (T < 0 || top_k < 1 || E < 1)
        return fail(MOE_ERR_INVALID_ARG, "moe_permute_align_static: bad T, top_k or E");
    const size_t need = moe_permute_workspace_size(T, top_k, E);
    if (need > kStaticScratchBytes)
        return fail(MOE_ERR_WORKSPACE_TOO_SMALL,
                    "moe_permute_align_static: this routing needs " + std::to_string(need) +
                        " bytes of scratch, more than the built-in " + std::to_string(kStaticScratchBytes) +
                        "; use moe_permute_align with a caller-provided workspace");
    void* scratch = nullptr;
    int rc = static_scratch(&scratch);
    if (rc != MOE_OK) return rc;
    return moe_permute_align(topk_ids, T, top_k, E, layout, block_m, max_tokens, x, x_dtype, K, x_out, rows_cap,
                             expert_counts, expert_offsets, row_route, route_row, scratch, kStaticScratchBytes,
                             err_word, stream);
}
