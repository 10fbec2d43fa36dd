// MXFP8 encoding helpers shared by the quantiser and the GEMM epilogues that
// emit MXFP8 directly, so that every producer of E4M3 codes + E8M0 scales
// makes the same decisions bit for bit.
//
// Scale code of a block from its maximum magnitude m, with integer arithmetic
// on the fp32 bits (exact, no logarithm): writing m = f * 2^p with f in [1, 2),
// the smallest c with m <= 448 * 2^c = 1.75 * 2^(c+8) is c = p - 8 when
// f <= 1.75 and c = p - 7 otherwise; code = clamp(c + 127, 0, 254), 0 when
// m == 0.  Elements are multiplied by 2^(127 - code) (a power of two, exact
// for every value that does not round to zero in E4M3) and converted with the
// hardware round-to-nearest-even saturating fp32 -> E4M3 conversion.
#pragma once

#include "common.cuh"

namespace moe {

MOE_DEVICE int mx_scale_code(float m) {
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

// Two fp32 values -> two E4M3 codes (lo in the low byte).
MOE_DEVICE uint16_t mx_cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

MOE_DEVICE float mx_pow2(int k) {   // 2^k for -149 <= k <= 127, exact
    if (k >= -126) return __uint_as_float(uint32_t(k + 127) << 23);
    return __uint_as_float(1u << (k + 149));
}

// The factor that maps a block with scale code `code` onto the E4M3 grid.
MOE_DEVICE float mx_inv_scale(int code) { return mx_pow2(127 - code); }

}  // namespace moe
