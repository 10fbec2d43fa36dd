// mxfp8_quantize_block32: one thread per block of 32 consecutive elements.
// The scale code is found with integer arithmetic on the fp32 bits of the
// block maximum m (exact, no logarithm): writing m = f * 2^p with f in [1, 2),
// the smallest c with m <= 448 * 2^c = 1.75 * 2^(c+8) is c = p - 8 when
// f <= 1.75 and c = p - 7 otherwise; code = clamp(c + 127, 0, 254), 0 when
// m == 0.  Elements are multiplied by 2^(127 - code) (a power of two, exact
// for every value that does not round to zero in E4M3) and converted with the
// hardware round-to-nearest-even saturating fp32 -> E4M3 conversion.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

MOE_DEVICE int scale_code_from_max(float m) {
    const uint32_t b = __float_as_uint(m);
    if (b == 0) return 0;
    int p;
    uint32_t frac;   // 23-bit fraction of the normalised significand
    const uint32_t ef = b >> 23;
    if (ef != 0) {
        p = int(ef) - 127;
        frac = b & 0x7FFFFFu;
    } else {   // subnormal: m = b * 2^-149
        const int msb = 31 - __clz(b);
        p = msb - 149;
        frac = (b << (23 - msb)) & 0x7FFFFFu;
    }
    const int c = (frac <= 0x600000u) ? p - 8 : p - 7;   // 0x600000 = 0.75 * 2^23
    return min(max(c + 127, 0), 254);
}

MOE_DEVICE uint16_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

MOE_DEVICE float pow2(int k) {   // 2^k for -149 <= k <= 127, exact
    if (k >= -126) return __uint_as_float(uint32_t(k + 127) << 23);
    return __uint_as_float(1u << (k + 149));
}

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
        const int code = scale_code_from_max(m);
        const float inv = pow2(127 - code);
        uint32_t packed[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t lo = cvt_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv);
            uint32_t hi = cvt_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv);
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
