// Device helpers shared by the kernels of libmoe_layer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_layer.h"

#define MOE_DEVICE __device__ __forceinline__

namespace moe {

constexpr int kWarp = 32;

// ---- element conversions -------------------------------------------------

MOE_DEVICE float bf16_bits_to_float(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }

// Round-to-nearest-even float -> bf16 bits (cvt.rn.bf16.f32; NaN stays NaN).
MOE_DEVICE uint16_t float_to_bf16_bits(float f) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}

// Two floats -> packed bf16x2 (lo in bits 0..15).
MOE_DEVICE uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <int DT>
MOE_DEVICE float load_as_float(const void* p, int64_t idx) {
    if constexpr (DT == MOE_F32) return static_cast<const float*>(p)[idx];
    else return bf16_bits_to_float(static_cast<const uint16_t*>(p)[idx]);
}

template <int DT>
MOE_DEVICE void store_from_float(void* p, int64_t idx, float v) {
    if constexpr (DT == MOE_F32) static_cast<float*>(p)[idx] = v;
    else static_cast<uint16_t*>(p)[idx] = float_to_bf16_bits(v);
}

// 8 consecutive elements <-> 8 floats, one 16-byte (bf16) or two 16-byte (f32) accesses.
template <int DT>
MOE_DEVICE void load8(const void* base, int64_t elem, float (&v)[8]) {
    if constexpr (DT == MOE_F32) {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem);
        float4 a = p[0], b = p[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        uint4 q = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem);
        uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
}

template <int DT>
MOE_DEVICE void store8(void* base, int64_t elem, const float (&v)[8]) {
    if constexpr (DT == MOE_F32) {
        float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + elem);
        p[0] = make_float4(v[0], v[1], v[2], v[3]);
        p[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
        uint4 q;
        q.x = pack_bf16x2(v[0], v[1]);
        q.y = pack_bf16x2(v[2], v[3]);
        q.z = pack_bf16x2(v[4], v[5]);
        q.w = pack_bf16x2(v[6], v[7]);
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + elem) = q;
    }
}

MOE_DEVICE void report(int32_t* err_word, int bit) {
    if (err_word) atomicOr(err_word, bit);
}

MOE_DEVICE float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// SiLU-and-mul with the fast exponential and division intrinsics (__expf, __fdividef): a few ulp from
// silu_mul, for epilogues where the full-precision division dominates the instruction count.  For g below
// about -87 the denominator overflows and the result is 0 (silu_mul gives a value below 1e-36 there).
MOE_DEVICE float silu_mul_fast(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

// ---- expert tile schedule -------------------------------------------------
//
// A grouped GEMM walks "tiles" that each belong to one expert.  The number of
// tiles of expert e is a function of its row count, so the list is built on
// the device from expert_counts (no host synchronisation): every CTA loads the
// counts into shared memory, takes an inclusive prefix sum of tiles per expert
// and maps a linear tile index to (expert, tile within expert) by binary
// search.  E <= kMaxExperts.

constexpr int kMaxExperts = 1024;

struct ExpertTable {
    int32_t tile_end[kMaxExperts];   // inclusive prefix of tiles per expert
    int32_t count[kMaxExperts];
    int32_t start[kMaxExperts];      // first row of the expert
    int32_t total;                   // tiles in all
};

// Block-wide build of the table.  `tiles_of(count)` gives the tiles of one
// expert.  Must be called by all threads of the block; ends with __syncthreads.
// Counts are clamped so that no expert reaches past its rows: the batched
// layout holds max_tokens rows per expert, the contiguous one rows_cap rows.
template <typename TilesOf>
__device__ void build_expert_table(ExpertTable& tab, int E, const int32_t* counts, const int32_t* offsets,
                                   int64_t max_tokens, int64_t rows_cap, TilesOf tiles_of) {
    __shared__ int32_t warp_sums[32];
    const int tid = threadIdx.x, nthr = blockDim.x;
    // each thread owns a contiguous run of experts so that a prefix over runs works
    const int per = (E + nthr - 1) / nthr;
    const int e0 = tid * per, e1 = min(E, e0 + per);
    int32_t local = 0;
    for (int e = e0; e < e1; ++e) {
        int64_t c = counts[e];
        const int64_t st = offsets ? int64_t(offsets[e]) : int64_t(e) * max_tokens;
        const int64_t room = offsets ? rows_cap - st : max_tokens;
        if (st < 0 || room < 0) c = 0;
        c = c < 0 ? 0 : (c > room ? room : c);
        tab.count[e] = int32_t(c);
        tab.start[e] = int32_t(st < 0 ? 0 : st);
        local += tiles_of(c);
    }
    // block exclusive scan of `local`
    const int lane = tid & 31, warp = tid >> 5, nwarps = (nthr + 31) >> 5;
    int32_t incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int32_t n = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += n;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int32_t s = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int32_t n = __shfl_up_sync(0xffffffffu, s, d);
            if (lane >= d) s += n;
        }
        warp_sums[lane] = s;   // inclusive over warps
    }
    __syncthreads();
    int32_t run = incl - local + (warp > 0 ? warp_sums[warp - 1] : 0);
    for (int e = e0; e < e1; ++e) {
        run += tiles_of(tab.count[e]);
        tab.tile_end[e] = run;
    }
    if (tid == nthr - 1) tab.total = run;
    __syncthreads();
}

// Expert owning linear tile `t` (t < total): first e with tile_end[e] > t.
MOE_DEVICE int find_expert(const ExpertTable& tab, int E, int32_t t) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (tab.tile_end[mid] > t) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

MOE_DEVICE int32_t tiles_before(const ExpertTable& tab, int e) { return e > 0 ? tab.tile_end[e - 1] : 0; }

}  // namespace moe
