// mxfp8_quantize_block32: one thread per block of 32 consecutive elements;
// the scale rule and the conversion are those of mx_codec.cuh.
#include "common.cuh"
#include "internal.h"
#include "mx_codec.cuh"

namespace moe {

namespace {

template <int DT>
__global__ void __launch_bounds__(256) mxfp8_kernel(const void* __restrict__ x, int64_t nblocks,
                                                    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
    for (int64_t b = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; b < nblocks;
         b += int64_t(gridDim.x) * blockDim.x) {
        float v[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float t[8];
            load8<DT>(x, b * 32 + q * 8, t);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[q * 8 + i] = t[i];
        }
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(v[i]));
        const int code = mx_scale_code(m);
        const float inv = mx_inv_scale(code);
        uint32_t packed[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t lo = mx_cvt_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv);
            uint32_t hi = mx_cvt_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv);
            packed[i] = lo | (hi << 16);
        }
        uint4* dst = reinterpret_cast<uint4*>(codes + b * 32);
        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        scales[b] = uint8_t(code);
    }
}

}  // namespace

cudaError_t launch_mxfp8_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, uint8_t* codes,
                                  uint8_t* scales, cudaStream_t s) {
    const int64_t nblocks = rows * (cols / 32);
    if (nblocks == 0) return cudaSuccess;
    int64_t grid = (nblocks + 255) / 256;
    const int64_t cap = int64_t(num_sms()) * 16;
    if (grid > cap) grid = cap;
    if (x_dtype == MOE_F32)
        mxfp8_kernel<MOE_F32><<<unsigned(grid), 256, 0, s>>>(x, nblocks, codes, scales);
    else
        mxfp8_kernel<MOE_BF16><<<unsigned(grid), 256, 0, s>>>(x, nblocks, codes, scales);
    return cudaGetLastError();
}

}  // namespace moe
