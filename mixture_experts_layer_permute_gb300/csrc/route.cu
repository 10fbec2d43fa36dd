// moe_topk_route: one warp per token, the E logits held in registers
// (E/32 per lane), top-k by repeated warp arg-max with the lower index
// winning ties, then softmax weights over the chosen (or all) logits.
#include "internal.h"
#include "route_device.cuh"

namespace moe {

namespace {

template <int PER_LANE>
__global__ void __launch_bounds__(256) topk_route_kernel(const float* __restrict__ logits, int64_t T, int E,
                                                         int k, int renorm, int32_t* __restrict__ ids,
                                                         float* __restrict__ weights) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    int id;
    float w;
    route_token<PER_LANE>(logits + t * E, E, k, renorm, lane, &id, &w);
    if (lane < k) {
        ids[t * k + lane] = id;
        weights[t * k + lane] = w;
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
