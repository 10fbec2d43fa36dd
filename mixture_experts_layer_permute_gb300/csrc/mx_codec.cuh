// MXFP8 helpers of the CUDA path: the encoding shared by the quantiser and the
// GEMM epilogues that emit MXFP8 directly, so that every producer of E4M3
// codes + E8M0 scales makes the same decisions bit for bit, and the decoding
// of E4M3 weights to bf16 used by the tcgen05 kernels (end of this file).
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

// ---- E4M3 weights decoded to bf16 for the kind::f16 MMA ----
//
// Placing an E4M3 code's sign in bf16 bit 15 and its exponent and mantissa in bits 10..4 gives exactly
// code * 2^-120 for normal, subnormal and zero codes alike; one bf16x2 multiply by 2^(scale-7) then yields
// code * 2^(scale-127).  mx_e4m3_factor gives that factor for scale code sc and whether the result still needs
// the second factor 2^120 (above sc = 134, 2^(sc-7) leaves bf16's range, so 2^(sc-127) is applied first).

// 4 E4M3 codes (one 32-bit word) -> 2 bf16x2 words (codes 0,1 and 2,3) times f1.
// prmt copies each code into the low byte of a 16-bit half and its sign into the high byte;
// shifting by 4 moves exponent+mantissa to bits 10..4 and the sign bits to 15..12 (and 19..16,
// outside the half); the mask keeps bits 15 and 10..4 of each half.
MOE_DEVICE void dequant4(uint32_t w, uint32_t f1, uint32_t& lo, uint32_t& hi) {
    uint32_t a, b;
    asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(a) : "r"(w));   // [sx(c1) c1 sx(c0) c0]
    asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(b) : "r"(w));   // [sx(c3) c3 sx(c2) c2]
    a = (a << 4) & 0x87F087F0u;
    b = (b << 4) & 0x87F087F0u;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(f1));
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(f1));
}

MOE_DEVICE uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

MOE_DEVICE uint32_t mx_e4m3_factor(uint32_t sc, bool& second) {
    second = sc > 134u;
    const uint32_t e1 = second ? sc : sc + 120u;
    return (e1 << 7) | (e1 << 23);
}

constexpr uint32_t kBf16x2Pow2_120 = (247u << 7) | (247u << 23);   // 2^120 in both halves

// Nonzero when a byte (scale code) of `quad` is above 134: its bit 7 set and its low 7 bits at least 7 (the
// per-byte sums stay below 256, so no carry crosses a byte).
MOE_DEVICE uint32_t mx_scale_above_134(uint32_t quad) {
    return ((quad & 0x7F7F7F7Fu) + 0x79797979u) & quad & 0x80808080u;
}

// mx_e4m3_factor of byte b of a scale word whose codes are all at most 134, from q120 = quad + 0x78787878
// (sc + 120 in each byte, no carry): byte b placed in bytes 1 and 3, shifted down by one bit, lands in both
// bf16 exponent fields.
MOE_DEVICE uint32_t mx_e4m3_factor_small(uint32_t q120, int b) {
    return __byte_perm(q120, 0u, 0x0404u | (uint32_t(b) << 4) | (uint32_t(b) << 12)) >> 1;
}

}  // namespace moe
