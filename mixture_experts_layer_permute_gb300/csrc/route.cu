// moe_topk_route: one warp per token, the E logits held in registers
// (E/32 per lane), top-k by repeated warp arg-max with the lower index
// winning ties, then softmax weights over the chosen (or all) logits.
#include <float.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

// a beats b: larger value, or equal value and smaller index.
MOE_DEVICE bool beats(float av, int ai, float bv, int bi) { return av > bv || (av == bv && ai < bi); }

template <int PER_LANE>
__global__ void __launch_bounds__(256) topk_route_kernel(const float* __restrict__ logits, int64_t T, int E,
                                                         int k, int renorm, int32_t* __restrict__ ids,
                                                         float* __restrict__ weights) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    const float* row = logits + t * E;
    float v[PER_LANE];
    uint32_t avail = 0;   // bit i: entry i of this lane is a candidate
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
        int e = i * 32 + lane;
        v[i] = e < E ? row[e] : -FLT_MAX;
        if (e < E) avail |= 1u << i;
    }
    int my_id = -1;
    float my_val = 0.f, lmax = 0.f, denom_sel = 0.f;
    for (int j = 0; j < k; ++j) {
        // lane-local best among available entries
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            if ((avail >> i) & 1u) {
                int e = i * 32 + lane;
                if (bi == 0x7fffffff || beats(v[i], e, bv, bi)) { bv = v[i]; bi = e; }
            }
        }
        // warp arg-max (value, then lower index)
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, d);
            int oi = __shfl_xor_sync(0xffffffffu, bi, d);
            if (oi != 0x7fffffff && (bi == 0x7fffffff || beats(ov, oi, bv, bi))) { bv = ov; bi = oi; }
        }
        if ((bi & 31) == lane) avail &= ~(1u << (bi >> 5));
        if (j == 0) lmax = bv;
        float p = expf(bv - lmax);
        denom_sel += p;            // same order on every lane
        if (lane == j) { my_id = bi; my_val = p; }
    }
    float denom = denom_sel;
    if (!renorm) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i)
            if (i * 32 + lane < E) s += expf(v[i] - lmax);
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) s += __shfl_xor_sync(0xffffffffu, s, d);
        denom = s;
    }
    if (lane < k) {
        ids[t * k + lane] = my_id;
        weights[t * k + lane] = my_val / denom;
    }
}

template <int PER_LANE>
cudaError_t launch(const float* logits, int64_t T, int E, int k, int renorm, int32_t* ids, float* w,
                   cudaStream_t s) {
    const int64_t threads = T * 32;
    const int64_t blocks = (threads + 255) / 256;
    topk_route_kernel<PER_LANE><<<unsigned(blocks), 256, 0, s>>>(logits, T, E, k, renorm, ids, w);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_topk_route(const float* logits, int64_t T, int E, int top_k, int renorm, int32_t* ids,
                              float* weights, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (E <= 32) return launch<1>(logits, T, E, top_k, renorm, ids, weights, s);
    if (E <= 64) return launch<2>(logits, T, E, top_k, renorm, ids, weights, s);
    if (E <= 128) return launch<4>(logits, T, E, top_k, renorm, ids, weights, s);
    if (E <= 256) return launch<8>(logits, T, E, top_k, renorm, ids, weights, s);
    if (E <= 512) return launch<16>(logits, T, E, top_k, renorm, ids, weights, s);
    return launch<32>(logits, T, E, top_k, renorm, ids, weights, s);
}

}  // namespace moe
