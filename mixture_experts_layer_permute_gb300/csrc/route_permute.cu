// moe_route_permute_align for small batches in one launch: routing, the
// stable expert-major placement and the row gather, which otherwise take three
// launches (route, permute, gather) whose fixed costs dominate at decode sizes.
//
// Every CTA routes all T tokens and ranks all routes itself, in shared memory
// (a few microseconds of redundant work on L2-resident logits), so no CTA ever
// waits for another.  CTA 0 alone writes ids, weights, counts, offsets and the
// two maps; each CTA then copies its share of the routed rows, 16-byte vectors
// spread over the whole grid.  The arithmetic is the route kernel's and the
// permute kernels' own (route_device.cuh, permute_device.cuh), so the results
// are bit-identical to the separate launches.
#include "internal.h"
#include "permute_device.cuh"
#include "route_device.cuh"

namespace moe {

namespace {

constexpr int kFusedMaxTokens = 128;        // at most 4 tokens per warp in the routing phase
constexpr int64_t kBytesPerCta = 32 << 10;  // gather share of one CTA

template <int PER_LANE>
__global__ void __launch_bounds__(kThreads) route_permute_kernel(
    const float* __restrict__ logits, int T, int E, int k, int renorm, int32_t* __restrict__ topk_ids,
    float* __restrict__ topk_weights, int layout, int block_m, int max_tokens, int32_t* counts, int32_t* offsets,
    int32_t* row_route, int32_t* route_row, const uint8_t* __restrict__ x, int64_t row_bytes,
    uint8_t* __restrict__ x_out, int32_t* err_word) {
    extern __shared__ __align__(16) uint8_t table[];   // [32][E]
    __shared__ SmemCommon sm;
    // expert of route r, then (once thread r has ranked it) its row; thread r alone touches entry r in between
    __shared__ int32_t route_s[kThreads];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = T * k;
    const bool lead = blockIdx.x == 0;
    for (int i = threadIdx.x; i < 32 * E; i += kThreads) table[i] = 0;
    for (int e = threadIdx.x; e < E; e += kThreads) sm.run[e] = 0;

    // 1. routing: one warp per token
    for (int t = warp; t < T; t += kThreads / 32) {
        int id;
        float w;
        route_token<PER_LANE>(logits + int64_t(t) * E, E, k, renorm, lane, &id, &w);
        if (lane < k) {
            route_s[t * k + lane] = id;
            if (lead) {
                topk_ids[t * k + lane] = id;
                topk_weights[t * k + lane] = w;
            }
        }
    }
    __syncthreads();

    // 2. placement: rank within the expert, expert layout, row of each route
    int e, rk;
    rank_round(route_s, threadIdx.x, R, E, table, err_word, lead, e, rk);
    absorb_round(table, sm.run, E);
    layout_experts(sm.run, sm.start, E, layout, block_m, max_tokens, counts, offsets, lead, sm.warp_buf);
    if (int(threadIdx.x) < R) {
        route_s[threadIdx.x] = int32_t(route_slot(e, rk, sm.start, layout, max_tokens));
        if (lead) place_route(threadIdx.x, e, rk, sm.start, layout, max_tokens, row_route, route_row, err_word);
    }
    for (int xe = blockIdx.x * (kThreads / 32) + warp; xe < E; xe += gridDim.x * (kThreads / 32))
        fill_padding(row_route, xe, sm.run, sm.start, layout == MOE_LAYOUT_CONTIGUOUS ? &sm.start[xe + 1] : nullptr,
                     layout, max_tokens, lane, 32);
    if (x_out == nullptr) return;
    __syncthreads();

    // 3. gather: vector i of route r goes to vector i of row slot(r); four vectors in flight per thread
    const int n16 = int(row_bytes / 16);
    const int total = R * n16;
    const int stride = int(gridDim.x) * kThreads;
    const uint4* src = reinterpret_cast<const uint4*>(x);
    uint4* dst = reinterpret_cast<uint4*>(x_out);
    for (int base = blockIdx.x * kThreads + threadIdx.x; base < total; base += 4 * stride) {
        uint4 v[4];
        int64_t to[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = base + u * stride;
            to[u] = -1;
            if (idx < total) {
                const int r = idx / n16, i = idx - r * n16;
                const int s = route_s[r];
                if (s >= 0) {
                    v[u] = src[int64_t(r / k) * n16 + i];
                    to[u] = int64_t(s) * n16 + i;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (to[u] >= 0) dst[to[u]] = v[u];
    }
}

template <int PER_LANE>
cudaError_t launch(const float* logits, int T, int E, int k, int renorm, int32_t* ids, float* w, int layout,
                   int block_m, int max_tokens, int32_t* counts, int32_t* offsets, int32_t* row_route,
                   int32_t* route_row, const void* x, int64_t row_bytes, void* x_out, int32_t* err_word,
                   cudaStream_t s) {
    int64_t grid = 1;
    if (x_out) {
        grid = (int64_t(T) * k * row_bytes + kBytesPerCta - 1) / kBytesPerCta;
        if (grid > num_sms()) grid = num_sms();
        if (grid < 1) grid = 1;
    }
    route_permute_kernel<PER_LANE><<<unsigned(grid), kThreads, size_t(32) * E, s>>>(
        logits, T, E, k, renorm, ids, w, layout, block_m, max_tokens, counts, offsets, row_route, route_row,
        static_cast<const uint8_t*>(x), row_bytes, static_cast<uint8_t*>(x_out), err_word);
    return cudaGetLastError();
}

}  // namespace

bool route_permute_fusable(int64_t T, int top_k, int64_t row_bytes) {
    return T >= 1 && T <= kFusedMaxTokens && T * top_k <= kThreads &&
           T * top_k * (row_bytes / 16) < (int64_t(1) << 31);
}

cudaError_t launch_route_permute(const float* logits, int64_t T, int E, int top_k, int renorm, int32_t* ids,
                                 float* weights, int layout, int block_m, int max_tokens, int32_t* counts,
                                 int32_t* offsets, int32_t* row_route, int32_t* route_row, const void* x,
                                 int64_t row_bytes, void* x_out, int32_t* err_word, cudaStream_t s) {
    const int t = int(T);
#define MOE_RP(P)                                                                                            \
    return launch<P>(logits, t, E, top_k, renorm, ids, weights, layout, block_m, max_tokens, counts, offsets, \
                     row_route, route_row, x, row_bytes, x_out, err_word, s)
    if (E <= 32) MOE_RP(1);
    if (E <= 64) MOE_RP(2);
    if (E <= 128) MOE_RP(4);
    if (E <= 256) MOE_RP(8);
    if (E <= 512) MOE_RP(16);
    MOE_RP(32);
#undef MOE_RP
}

}  // namespace moe
