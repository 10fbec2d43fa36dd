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
// held until the process exits.  Its device address is looked up with
// cudaGetSymbolAddress on the first call in each CUDA context of a device
// (so make that first call before any stream capture) and kept for that
// context only: after cudaDeviceReset, or when the primary context is
// released and created again, the module is loaded anew and the next call
// looks the address up again instead of using a stale one.  All calls
// share the one array, so two calls that overlap on the GPU (different
// streams, or different host threads on one device) race on it and must be
// serialised by the caller.  Nothing in the scratch has to start at zero:
// each call writes every entry it later reads.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>
#include <string>

#include "internal.h"
#include "moe_layer.h"

namespace moe {

namespace {

constexpr size_t kStaticScratchBytes = size_t(2) << 20;   // 2 MiB

static __device__ __align__(256) unsigned char g_permute_scratch[kStaticScratchBytes];

// Identity of the calling thread's current CUDA context (cuCtxGetId, taken through the runtime's driver entry
// point table); 0 when there is no current context or the driver cannot say.
unsigned long long current_context_id() {
    using GetCurrentFn = int (*)(void**);
    using GetIdFn = int (*)(void*, unsigned long long*);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(p);
    });
    if (!get_current || !get_id) return 0;
    void* ctx = nullptr;
    if (get_current(&ctx) != 0 || !ctx) return 0;
    unsigned long long id = 0;
    return get_id(ctx, &id) == 0 ? id : 0;
}

// Device address of g_permute_scratch in the current context.  It is cached per device together with the
// context it was taken in; a call from another context (a reset device, a re-created primary context) looks it
// up again.  Without a context id to compare, every call looks it up (a host-side table read once the module
// is loaded).
int static_scratch(void** out) {
    static std::mutex mu;
    static void* addr[64] = {};
    static unsigned long long ctx_of[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(MOE_ERR_LAUNCH, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(MOE_ERR_UNSUPPORTED, "moe_permute_align_static: device index >= 64");
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long ctx = current_context_id();
    if (ctx != 0 && addr[dev] && ctx_of[dev] == ctx) {
        *out = addr[dev];
        return MOE_OK;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess || !p)
        return fail(MOE_ERR_LAUNCH, std::string("cudaGetSymbolAddress(g_permute_scratch): ") + cudaGetErrorString(e));
    addr[dev] = p;
    ctx_of[dev] = current_context_id();   // the look-up made the context current if none was
    *out = p;
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
    if (T < 0 || top_k < 1 || top_k > 1024 || E < 1 || E > 1024 || T > (int64_t(INT32_MAX) / top_k))
        return fail(MOE_ERR_INVALID_ARG, "moe_permute_align_static: bad T, top_k or E (T*top_k must stay below 2^31, "
                                         "top_k and E in [1, 1024])");
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
