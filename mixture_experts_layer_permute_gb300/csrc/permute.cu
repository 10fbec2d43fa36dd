// moe_permute_align: counts routes per expert, lays experts out one after the
// other (padded to block_m rows in the contiguous layout, at e*max_tokens in
// the batched one) and places each route at (expert start + its rank among
// the earlier routes of the same expert).  The rank is computed without any
// sort: routes are taken 1024 at a time (one per thread, route index order);
// __match_any_sync groups the lanes of a warp that share an expert, a byte
// table [warp][expert] in shared memory holds each warp's group sizes, and a
// thread's rank is the group sizes of the earlier warps plus the earlier lanes
// of its own group.  Counts carried across rounds and across CTAs (a per-chunk
// histogram in the workspace) extend the rank to any number of routes, so the
// placement is the stable order of the routes -- unique, run-to-run identical.
#include "internal.h"
#include "permute_device.cuh"

namespace moe {

namespace {

constexpr int kMaxChunks = 64;

// ---- single CTA: routes <= 1024 -----------------------------------------
__global__ void __launch_bounds__(kThreads) permute_single_kernel(
    const int32_t* __restrict__ ids, int64_t R, int E, int layout, int block_m, int max_tokens,
    int32_t* counts, int32_t* offsets, int32_t* row_route, int32_t* route_row, int32_t* err_word) {
    extern __shared__ __align__(16) uint8_t table[];   // [32][E]
    __shared__ SmemCommon sm;
    for (int i = threadIdx.x; i < 32 * E; i += kThreads) table[i] = 0;
    for (int e = threadIdx.x; e < E; e += kThreads) sm.run[e] = 0;
    __syncthreads();
    int e, rk;
    rank_round(ids, threadIdx.x, R, E, table, err_word, true, e, rk);
    absorb_round(table, sm.run, E);
    layout_experts(sm.run, sm.start, E, layout, block_m, max_tokens, counts, offsets, true, sm.warp_buf);
    if (threadIdx.x < R)
        place_route(threadIdx.x, e, rk, sm.start, layout, max_tokens, row_route, route_row, err_word);
    // padding rows: one warp per expert
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int x = warp; x < E; x += kThreads / 32)
        fill_padding(row_route, x, sm.run, sm.start, layout == MOE_LAYOUT_CONTIGUOUS ? &sm.start[x + 1] : nullptr,
                     layout, max_tokens, lane, 32);
}

// ---- several CTAs ----------------------------------------------------------
// Pass 1: rank of each route within its chunk, per-chunk expert histogram.
__global__ void __launch_bounds__(kThreads) permute_chunk_kernel(const int32_t* __restrict__ ids, int64_t R, int E,
                                                                 int rounds, int32_t* chunk_counts,
                                                                 int32_t* ranks, int32_t* err_word) {
    extern __shared__ __align__(16) uint8_t table[];
    __shared__ int32_t run[kMaxExperts];
    for (int i = threadIdx.x; i < 32 * E; i += kThreads) table[i] = 0;
    for (int e = threadIdx.x; e < E; e += kThreads) run[e] = 0;
    __syncthreads();
    const int64_t base = int64_t(blockIdx.x) * rounds * kThreads;
    for (int q = 0; q < rounds; ++q) {
        const int64_t r = base + int64_t(q) * kThreads + threadIdx.x;
        int e, rk;
        rank_round(ids, r, R, E, table, err_word, true, e, rk);
        if (r < R) ranks[r] = e >= 0 ? run[e] + rk : -1;
        absorb_round(table, run, E);
    }
    for (int e = threadIdx.x; e < E; e += kThreads) chunk_counts[int64_t(blockIdx.x) * E + e] = run[e];
}

// Pass 2: expert layout from the histograms, then each route's row.
__global__ void __launch_bounds__(kThreads) permute_scatter_kernel(
    const int32_t* __restrict__ ids, int64_t R, int E, int rounds, int nchunks, const int32_t* chunk_counts,
    const int32_t* ranks, int layout, int block_m, int max_tokens, int32_t* counts, int32_t* offsets,
    int32_t* row_route, int32_t* route_row, int32_t* err_word) {
    __shared__ SmemCommon sm;
    __shared__ int32_t before[kMaxExperts];
    for (int e = threadIdx.x; e < E; e += kThreads) {
        int32_t tot = 0, pre = 0;
        for (int c = 0; c < nchunks; ++c) {
            int32_t v = chunk_counts[int64_t(c) * E + e];
            if (c < int(blockIdx.x)) pre += v;
            tot += v;
        }
        sm.run[e] = tot;
        before[e] = pre;
    }
    __syncthreads();
    layout_experts(sm.run, sm.start, E, layout, block_m, max_tokens, counts, offsets, blockIdx.x == 0,
                   sm.warp_buf);
    const int64_t base = int64_t(blockIdx.x) * rounds * kThreads;
    for (int q = 0; q < rounds; ++q) {
        const int64_t r = base + int64_t(q) * kThreads + threadIdx.x;
        if (r >= R) break;
        int v = ids[r];
        int e = (v >= 0 && v < E) ? v : -1;
        int rk = e >= 0 ? ranks[r] + before[e] : 0;
        place_route(r, e, rk, sm.start, layout, max_tokens, row_route, route_row, err_word);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int x = blockIdx.x * (kThreads / 32) + warp; x < E; x += gridDim.x * (kThreads / 32))
        fill_padding(row_route, x, sm.run, sm.start, layout == MOE_LAYOUT_CONTIGUOUS ? &sm.start[x + 1] : nullptr,
                     layout, max_tokens, lane, 32);
}

// ---- gather x rows into the permuted layout --------------------------------
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint8_t* __restrict__ x, int64_t row_bytes,
                                                          const int32_t* __restrict__ row_route, int top_k,
                                                          const int32_t* offsets, int E, int64_t rows_cap,
                                                          uint8_t* __restrict__ x_out) {
    const int64_t s = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t rows = offsets ? int64_t(offsets[E]) : rows_cap;
    if (s >= rows) return;
    const int r = row_route[s];
    if (r < 0) return;
    const uint4* src = reinterpret_cast<const uint4*>(x + int64_t(r / top_k) * row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(x_out + s * row_bytes);
    const int n = int(row_bytes / 16);   // vectors per row (the host keeps a row under 2^31 bytes)
    int i = lane;
#pragma unroll 1
    for (; i + 96 < n; i += 128) {   // four vectors in flight per lane
        const uint4 a = src[i], b = src[i + 32], c = src[i + 64], d = src[i + 96];
        dst[i] = a;
        dst[i + 32] = b;
        dst[i + 64] = c;
        dst[i + 96] = d;
    }
#pragma unroll 1
    for (; i < n; i += 32) dst[i] = src[i];
}

struct Plan {
    int64_t R;
    int rounds;
    int nchunks;
};

Plan plan_for(int64_t T, int top_k) {
    Plan p;
    p.R = T * top_k;
    p.rounds = int((p.R + int64_t(kThreads) * kMaxChunks - 1) / (int64_t(kThreads) * kMaxChunks));
    if (p.rounds < 1) p.rounds = 1;
    p.nchunks = int((p.R + int64_t(p.rounds) * kThreads - 1) / (int64_t(p.rounds) * kThreads));
    if (p.nchunks < 1) p.nchunks = 1;
    return p;
}

}  // namespace

size_t permute_workspace_bytes(int64_t T, int top_k, int E) {
    Plan p = plan_for(T, top_k);
    size_t a = size_t(p.nchunks) * size_t(E) * sizeof(int32_t);
    a = (a + 255) / 256 * 256;
    return a + size_t(p.R) * sizeof(int32_t) + 256;
}

cudaError_t launch_permute(const int32_t* ids, int64_t T, int top_k, int E, int layout, int block_m,
                           int max_tokens, int32_t* counts, int32_t* offsets, int32_t* row_route,
                           int32_t* route_row, void* ws, int32_t* err_word, cudaStream_t s) {
    Plan p = plan_for(T, top_k);
    const size_t table_bytes = size_t(32) * E;
    if (p.R <= kThreads) {
        permute_single_kernel<<<1, kThreads, table_bytes, s>>>(ids, p.R, E, layout, block_m, max_tokens, counts,
                                                               offsets, row_route, route_row, err_word);
        return cudaGetLastError();
    }
    int32_t* chunk_counts = static_cast<int32_t*>(ws);
    size_t a = size_t(p.nchunks) * size_t(E) * sizeof(int32_t);
    a = (a + 255) / 256 * 256;
    int32_t* ranks = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + a);
    permute_chunk_kernel<<<p.nchunks, kThreads, table_bytes, s>>>(ids, p.R, E, p.rounds, chunk_counts, ranks,
                                                                  err_word);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    permute_scatter_kernel<<<p.nchunks, kThreads, 0, s>>>(ids, p.R, E, p.rounds, p.nchunks, chunk_counts, ranks,
                                                          layout, block_m, max_tokens, counts, offsets, row_route,
                                                          route_row, err_word);
    return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* x, int esize, int64_t K, const int32_t* row_route, int top_k,
                               const int32_t* offsets, int E, int64_t rows_cap, void* x_out, cudaStream_t s) {
    if (rows_cap == 0) return cudaSuccess;
    const int64_t blocks = (rows_cap * 32 + 255) / 256;
    gather_rows_kernel<<<unsigned(blocks), 256, 0, s>>>(static_cast<const uint8_t*>(x), K * esize, row_route,
                                                        top_k, offsets, E, rows_cap,
                                                        static_cast<uint8_t*>(x_out));
    return cudaGetLastError();
}

}  // namespace moe
