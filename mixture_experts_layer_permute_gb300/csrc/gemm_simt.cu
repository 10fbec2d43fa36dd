// CUDA-core grouped GEMMs (fp32 FMA).  This is the path for fp32 layers --
// tensor-core tf32 would not hold a 1e-5 relative tolerance -- and for shapes
// the tcgen05 tiles do not cover.  Activations are F32, BF16 or MXFP8 (E4M3
// codes + E8M0 scales, with MXFP8 weights); weights F32, BF16 or MXFP8.  A CTA computes a 64 x 64 tile of
// C = A[rows of one expert] * B^T[64 weight rows] in 16-wide k steps staged
// through shared memory; each of the 256 threads owns a 4 x 4 block of C.
//   GEMM 1: the 64 weight rows are the gate rows and the up rows of 32 units,
//           and the epilogue writes h = silu(gate) * up.
//   GEMM 2: the 64 weight rows are 64 output columns; the epilogue scales by
//           the route weight and writes the (token, slot) row of the route.
// Tiles are listed per expert on the device (ExpertTable), so the launch needs
// no host copy of the counts.
#include "common.cuh"
#include "internal.h"
#include "mx_codec.cuh"

namespace moe {

namespace {

constexpr int BM = 64, BN = 64, BK = 16;

MOE_DEVICE float e4m3_to_float(uint8_t c) {
    const uint32_t s = uint32_t(c & 0x80) << 24;
    const uint32_t e = (c >> 3) & 0xF, m = c & 7;
    if (e == 0) return __uint_as_float(s | __float_as_uint(float(m) * 0.001953125f));   // m * 2^-9
    if (e == 15 && m == 7) return __uint_as_float(0x7FC00000u);
    return __uint_as_float(s | ((e + 120u) << 23) | (m << 20));
}

MOE_DEVICE float e8m0_to_float(uint8_t c) {   // 2^(c-127); c in [1, 254] is a normal float
    if (c == 0) return __uint_as_float(0x00400000u);   // 2^-127
    if (c == 255) return __uint_as_float(0x7FC00000u);
    return __uint_as_float(uint32_t(c) << 23);
}

template <int WDT>
MOE_DEVICE float load_weight(const void* w, const uint8_t* scale, int64_t row, int64_t col, int64_t ncols) {
    const int64_t idx = row * ncols + col;
    if constexpr (WDT == MOE_E4M3) {
        const float v = e4m3_to_float(static_cast<const uint8_t*>(w)[idx]);
        return v * e8m0_to_float(scale[row * (ncols / 32) + col / 32]);
    } else {
        return load_as_float<WDT>(w, idx);
    }
}

// Row of W1[e] holding gate (half 0) or up (half 1) of unit i.
MOE_DEVICE int64_t w1_row(int w1_layout, int64_t I, int half, int64_t i) {
    if (w1_layout == MOE_W1_GATE_UP) return half * I + i;
    return (i / 16) * 32 + half * 16 + (i % 16);
}

template <int GEMM, int ADT, int WDT, int ODT>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs g) {
    __shared__ ExpertTable tab;
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    __shared__ float Cs[GEMM == 1 ? BM : 1][BN + 1];

    build_expert_table(tab, g.E, g.counts, g.offsets, g.max_tokens, g.rows_cap,
                       [](int32_t c) { return (c + BM - 1) / BM; });
    const int32_t t = blockIdx.x;
    if (t >= tab.total) return;
    const int e = find_expert(tab, g.E, t);
    const int32_t mt = t - tiles_before(tab, e);
    const int64_t row0 = int64_t(tab.start[e]) + int64_t(mt) * BM;
    const int valid = min(BM, tab.count[e] - mt * BM);

    const int64_t kdim = GEMM == 1 ? g.K : g.I;           // contraction length
    const int64_t wrows = GEMM == 1 ? 2 * g.I : g.K;      // weight rows per expert
    const int64_t wbase_row = int64_t(e) * wrows;
    const int64_t n0 = int64_t(blockIdx.y) * (GEMM == 1 ? BN / 2 : BN);   // units (1) or columns (2)
    const int64_t ncols_out = GEMM == 1 ? g.I : g.K;

    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    float acc[4][4] = {};

    // This thread's 4 A and 4 B elements of the k-step at k0 (A: 64 rows x 16 k; B: 64 weight rows x 16 k).
    auto load_step = [&](int64_t k0, float (&ra)[4], float (&rb)[4]) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int idx = tid + q * 256, r = idx / BK, kk = idx % BK;
            float v = 0.f;
            if (r < valid) {
                if constexpr (ADT == MOE_E4M3) v = load_weight<MOE_E4M3>(g.a, g.a_scale, row0 + r, k0 + kk, kdim);
                else v = load_as_float<ADT>(g.a, (row0 + r) * kdim + k0 + kk);
            }
            ra[q] = v;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int idx = tid + q * 256, c = idx / BK, kk = idx % BK;
            float v = 0.f;
            int64_t wr;
            bool ok;
            if constexpr (GEMM == 1) {
                const int64_t unit = n0 + (c % 32);
                ok = unit < g.I;
                wr = w1_row(g.w1_layout, g.I, c / 32, unit);
            } else {
                wr = n0 + c;
                ok = wr < g.K;
            }
            if (ok) v = load_weight<WDT>(g.w, g.w_scale, wbase_row + wr, k0 + kk, kdim);
            rb[q] = v;
        }
    };

    // The k-steps' loads are issued PF steps ahead into registers, so a small layer (few k-steps, nothing in
    // cache) waits for memory once per PF steps instead of once per step; the sums run in the same order.
    constexpr int PF = 4;
    float ra[PF][4], rb[PF][4];
#pragma unroll
    for (int f = 0; f < PF; ++f)
        if (int64_t(f) * BK < kdim) load_step(int64_t(f) * BK, ra[f], rb[f]);
    for (int64_t k0 = 0; k0 < kdim; k0 += PF * BK) {
#pragma unroll
        for (int f = 0; f < PF; ++f) {
            const int64_t ks = k0 + int64_t(f) * BK;
            if (ks >= kdim) break;                         // the same for every thread of the block
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int idx = tid + q * 256;
                As[idx % BK][idx / BK] = ra[f][q];
                Bs[idx % BK][idx / BK] = rb[f][q];
            }
            __syncthreads();
            if (ks + PF * BK < kdim) load_step(ks + PF * BK, ra[f], rb[f]);   // refill this slot
#pragma unroll
            for (int kk = 0; kk < BK; ++kk) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) { a[i] = As[kk][ty * 4 + i]; b[i] = Bs[kk][tx * 4 + i]; }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
            __syncthreads();
        }
    }

    if constexpr (GEMM == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) Cs[ty * 4 + i][tx * 4 + j] = acc[i][j];
        __syncthreads();
        if constexpr (ODT == MOE_E4M3) {
            // MXFP8 h: the tile's 32 units (n0 % 32 == 0, I % 32 == 0) are one scale block of each row; one
            // thread per row rounds h to bf16, finds the block maximum and writes 32 codes and the scale
            const int r = tid;
            if (r < BM && r < valid && n0 + 32 <= g.I) {
                float hv[32];
                float m = 0.f;
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    hv[u] = bf16_bits_to_float(float_to_bf16_bits(silu_mul(Cs[r][u], Cs[r][u + 32])));
                    m = fmaxf(m, fabsf(hv[u]));
                }
                const int code = mx_scale_code(m);
                const float inv = mx_inv_scale(code);
                uint32_t packed[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t lo = mx_cvt_e4m3x2(hv[4 * i] * inv, hv[4 * i + 1] * inv);
                    const uint32_t hi = mx_cvt_e4m3x2(hv[4 * i + 2] * inv, hv[4 * i + 3] * inv);
                    packed[i] = lo | (hi << 16);
                }
                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(g.out) + (row0 + r) * g.I + n0);
                dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                g.out_scale[(row0 + r) * (g.I / 32) + n0 / 32] = uint8_t(code);
            }
        } else {
            for (int idx = tid; idx < BM * (BN / 2); idx += 256) {
                const int r = idx / (BN / 2), u = idx % (BN / 2);
                const int64_t unit = n0 + u;
                if (r < valid && unit < g.I)
                    store_from_float<ODT>(g.out, (row0 + r) * ncols_out + unit, silu_mul(Cs[r][u], Cs[r][u + 32]));
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = ty * 4 + i;
            if (r >= valid) continue;
            const int64_t row = row0 + r;
            int64_t dst_row;
            float wt = 1.f;
            if (g.layout == MOE_LAYOUT_CONTIGUOUS) {
                const int32_t route = g.row_route[row];
                if (route < 0 || route >= g.out_rows) continue;
                dst_row = route;
                if (g.route_w) wt = g.route_w[route];
            } else {
                dst_row = row;
                if (g.route_w) wt = g.route_w[row];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t col = n0 + tx * 4 + j;
                if (col < g.K) store_from_float<ODT>(g.out, dst_row * g.K + col, wt * acc[i][j]);
            }
        }
    }
}

template <int GEMM, int ADT, int WDT>
cudaError_t launch3(const GemmArgs& g, dim3 grid, cudaStream_t s) {
    if constexpr (GEMM == 1) {
        if (g.out_dtype == MOE_E4M3) {
            gemm_simt_kernel<GEMM, ADT, WDT, MOE_E4M3><<<grid, 256, 0, s>>>(g);
            return cudaGetLastError();
        }
    }
    if (g.out_dtype == MOE_F32) gemm_simt_kernel<GEMM, ADT, WDT, MOE_F32><<<grid, 256, 0, s>>>(g);
    else gemm_simt_kernel<GEMM, ADT, WDT, MOE_BF16><<<grid, 256, 0, s>>>(g);
    return cudaGetLastError();
}

template <int GEMM, int ADT>
cudaError_t launch2(const GemmArgs& g, dim3 grid, cudaStream_t s) {
    if (g.w_dtype == MOE_F32) return launch3<GEMM, ADT, MOE_F32>(g, grid, s);
    if (g.w_dtype == MOE_BF16) return launch3<GEMM, ADT, MOE_BF16>(g, grid, s);
    return launch3<GEMM, ADT, MOE_E4M3>(g, grid, s);
}

template <int GEMM>
cudaError_t launch1(const GemmArgs& g, dim3 grid, cudaStream_t s) {
    if (g.a_dtype == MOE_F32) return launch2<GEMM, MOE_F32>(g, grid, s);
    if (g.a_dtype == MOE_E4M3) return launch3<GEMM, MOE_E4M3, MOE_E4M3>(g, grid, s);   // MXFP8 x MXFP8
    return launch2<GEMM, MOE_BF16>(g, grid, s);
}

}  // namespace

cudaError_t launch_gemm_simt(const GemmArgs& g, cudaStream_t s) {
    // upper bound on the tiles: sum_e ceil(count_e / 64)
    int64_t mtiles;
    if (g.layout == MOE_LAYOUT_CONTIGUOUS) mtiles = (g.rows_cap + BM - 1) / BM + g.E;
    else mtiles = int64_t(g.E) * ((g.max_tokens + BM - 1) / BM);
    if (mtiles == 0) return cudaSuccess;
    const int64_t ntiles = g.gemm == 1 ? (g.I + BN / 2 - 1) / (BN / 2) : (g.K + BN - 1) / BN;
    const dim3 grid(static_cast<unsigned>(mtiles), static_cast<unsigned>(ntiles));
    return g.gemm == 1 ? launch1<1>(g, grid, s) : launch1<2>(g, grid, s);
}

}  // namespace moe
