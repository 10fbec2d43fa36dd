// The stable placement of routes into expert-major rows, shared by the
// permute kernels and the fused route + permute kernel.  Routes are taken
// 1024 at a time (one per thread, in route-index order); __match_any_sync
// groups the lanes of a warp that share an expert, a byte table
// [warp][expert] in shared memory holds each warp's group sizes, and a
// thread's rank is the group sizes of the earlier warps plus the earlier lanes
// of its own group.
#pragma once

#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;   // threads of every permute CTA (one route each per round)

// Exclusive prefix sum over the block (blockDim.x == kThreads); returns the
// exclusive value of `v` and writes the total to *total.
__device__ int block_exclusive_scan(int v, int* warp_buf, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += n;
    }
    if (lane == 31) warp_buf[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int s = warp_buf[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, s, d);
            if (lane >= d) s += n;
        }
        warp_buf[lane] = s;
    }
    __syncthreads();
    int excl = incl - v + (warp > 0 ? warp_buf[warp - 1] : 0);
    *total = warp_buf[31];
    __syncthreads();
    return excl;
}

// One round: thread tid takes route r (r < R) and returns its expert (-1 when
// skipped) and its rank among the routes of the round with the same expert and
// a smaller index.  `table` ([32][E] bytes) must be zero on entry; on return it
// holds each warp's per-expert counts (the caller sums and clears it).
__device__ void rank_round(const int32_t* __restrict__ ids, int64_t r, int64_t R, int E, uint8_t* table,
                           int32_t* err_word, bool report_errors, int& e_out, int& rank_out) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int e = -1;
    if (r < R) {
        int v = ids[r];
        if (v >= 0 && v < E) e = v;
        else if (v != -1 && report_errors) report(err_word, MOE_DEVERR_ID_RANGE);
    }
    const unsigned mask = __match_any_sync(0xffffffffu, e);
    int rk = __popc(mask & ((1u << lane) - 1u));
    if (e >= 0 && rk == 0) table[warp * E + e] = uint8_t(__popc(mask));
    __syncthreads();
    if (e >= 0) {
        for (int w = 0; w < warp; ++w) rk += table[w * E + e];
    }
    e_out = e;
    rank_out = rk;
}

// Sums the round's table into run[e] and clears the table (all threads).
__device__ void absorb_round(uint8_t* table, int32_t* run, int E) {
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads) {
        int s = 0;
        for (int w = 0; w < 32; ++w) s += table[w * E + e];
        run[e] += s;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 32 * E; i += kThreads) table[i] = 0;
    __syncthreads();
}

// Given total[e], computes start[e] (row of the expert's first route) and
// writes counts/offsets when `write` is set.
__device__ void layout_experts(const int32_t* total, int32_t* start, int E, int layout, int block_m, int max_tokens,
                               int32_t* counts, int32_t* offsets, bool write, int* warp_buf) {
    // E <= kThreads: one expert per thread
    const int e = threadIdx.x;
    int c = e < E ? total[e] : 0;
    if (layout == MOE_LAYOUT_CONTIGUOUS) {
        int padded = (c + block_m - 1) / block_m * block_m;
        int all;
        int ex = block_exclusive_scan(padded, warp_buf, &all);
        if (e < E) start[e] = ex;
        if (e == 0) start[E] = all;
        if (write) {
            if (e < E) { counts[e] = c; offsets[e] = ex; }
            if (e == 0) offsets[E] = all;
        }
    } else {
        if (e < E) start[e] = e * max_tokens;
        if (e == 0) start[E] = E * max_tokens;
        if (write) {
            if (e < E) { counts[e] = min(c, max_tokens); offsets[e] = e * max_tokens; }
            if (e == 0) offsets[E] = E * max_tokens;
        }
    }
    __syncthreads();
}

// Writes -1 to the rows of expert e that hold no route.
__device__ void fill_padding(int32_t* row_route, int e, const int32_t* total, const int32_t* start,
                             const int32_t* offsets_next, int layout, int max_tokens, int lane0, int stride) {
    int c = total[e];
    int64_t s0, s1;
    if (layout == MOE_LAYOUT_CONTIGUOUS) {
        s0 = int64_t(start[e]) + c;
        s1 = offsets_next ? int64_t(offsets_next[0]) : s0;
    } else {
        s0 = int64_t(start[e]) + min(c, max_tokens);
        s1 = int64_t(start[e]) + max_tokens;
    }
    for (int64_t s = s0 + lane0; s < s1; s += stride) row_route[s] = -1;
}

__device__ void place_route(int64_t r, int e, int rank, const int32_t* start, int layout, int max_tokens,
                            int32_t* row_route, int32_t* route_row, int32_t* err_word) {
    if (e < 0) { route_row[r] = -1; return; }
    if (layout == MOE_LAYOUT_BATCHED && rank >= max_tokens) {
        report(err_word, MOE_DEVERR_CAPACITY);
        route_row[r] = -1;
        return;
    }
    int64_t s = int64_t(start[e]) + rank;
    row_route[s] = int32_t(r);
    route_row[r] = int32_t(s);
}

struct SmemCommon {
    int32_t run[kMaxExperts];
    int32_t start[kMaxExperts + 1];
    int warp_buf[32];
};

// The row of a route of expert e (>= 0) with the given rank, or -1 when the
// batched layout's capacity drops it (the same decision as place_route).
MOE_DEVICE int64_t route_slot(int e, int rank, const int32_t* start, int layout, int max_tokens) {
    if (e < 0 || (layout == MOE_LAYOUT_BATCHED && rank >= max_tokens)) return -1;
    return int64_t(start[e]) + rank;
}

}  // namespace
}  // namespace moe
