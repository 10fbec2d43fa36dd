// moe_unpermute_topk_reduce and moe_batched_weight_reduce: HBM-bound
// elementwise passes.  Each thread owns 8 consecutive elements of one output
// row (one 16-byte bf16 vector), reads the top_k slot rows in increasing j and
// sums in fp32 in that fixed order, so the result is bit-identical run to run.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

// Raw 16-byte (bf16) or 32-byte (f32) vector of 8 elements.
template <int DT>
struct Vec8 {
    uint4 a, b;
};

template <int DT>
MOE_DEVICE Vec8<DT> ld_vec8(const void* base, int64_t elem) {
    Vec8<DT> v;
    if constexpr (DT == MOE_F32) {
        const uint4* p = reinterpret_cast<const uint4*>(static_cast<const float*>(base) + elem);
        v.a = p[0];
        v.b = p[1];
    } else {
        v.a = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem);
        v.b = make_uint4(0, 0, 0, 0);
    }
    return v;
}

template <int DT>
MOE_DEVICE void unpack8(const Vec8<DT>& v, float (&f)[8]) {
    if constexpr (DT == MOE_F32) {
        const uint32_t w[8] = {v.a.x, v.a.y, v.a.z, v.a.w, v.b.x, v.b.y, v.b.z, v.b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(w[i]);
    } else {
        const uint32_t w[4] = {v.a.x, v.a.y, v.a.z, v.a.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
}

// Slots are taken 8 at a time: their ids and weights are read first, then all 8 row vectors are
// requested before any is used, and the products are added in increasing j (the order, and so the
// result, does not depend on the batching).
// ROWS = false: slot (t, j) is valid when 0 <= ids[t,j] < lim (= E) and its row is t*top_k + j.
// ROWS = true:  `ids` is route_row, slot (t, j) reads row ids[t,j] when 0 <= ids[t,j] < lim (= rows);
//               entries other than -1 outside [0, rows) set MOE_DEVERR_ID_RANGE.
template <int YDT, int ODT, bool ROWS>
__global__ void __launch_bounds__(256) topk_reduce_kernel(const void* __restrict__ y,
                                                          const int32_t* __restrict__ ids,
                                                          const float* __restrict__ w, int64_t T, int top_k,
                                                          int64_t lim, int64_t K, void* __restrict__ out,
                                                          int32_t* err_word) {
    // grid: x over the 8-element column vectors of a row, y over output rows (no index division)
    const int64_t vec = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (vec >= K / 8) return;
    const int64_t col = vec * 8;
    for (int64_t t = blockIdx.y; t < T; t += gridDim.y) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j0 = 0; j0 < top_k; j0 += 8) {
            int e[8];
            float wj[8];
            Vec8<YDT> raw[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = j0 + u;
                e[u] = j < top_k ? ids[t * top_k + j] : -1;
                wj[u] = (w && j < top_k) ? w[t * top_k + j] : 1.0f;
            }
            if constexpr (ROWS) {
                // one thread per token row reports a bad row index
                if (vec == 0 && err_word) {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (e[u] < -1 || e[u] >= lim) report(err_word, MOE_DEVERR_ID_RANGE);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (e[u] >= 0 && e[u] < lim) {
                    const int64_t row = ROWS ? int64_t(e[u]) : t * top_k + j0 + u;
                    raw[u] = ld_vec8<YDT>(y, row * K + col);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (e[u] < 0 || e[u] >= lim) continue;
                float v[8];
                unpack8<YDT>(raw[u], v);
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] = fmaf(wj[u], v[q], acc[q]);
            }
        }
        store8<ODT>(out, t * K + col, acc);
    }
}

template <int YDT, int ODT>
__global__ void __launch_bounds__(256) batched_weight_kernel(const void* __restrict__ y,
                                                             const int32_t* __restrict__ counts,
                                                             const float* __restrict__ w, int E, int max_tokens,
                                                             int64_t K, void* out) {
    const int64_t vec = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (vec >= K / 8) return;
    const int64_t col = vec * 8;
    const int rows = E * max_tokens;   // the host keeps E * max_tokens below 2^31
    for (int row = blockIdx.y; row < rows; row += gridDim.y) {
        const int e = row / max_tokens, q = row - e * max_tokens;
        if (q >= counts[e]) continue;
        const float wr = w ? w[row] : 1.0f;
        float v[8];
        load8<YDT>(y, int64_t(row) * K + col, v);
#pragma unroll
        for (int c = 0; c < 8; ++c) v[c] = wr * v[c];
        store8<ODT>(out, int64_t(row) * K + col, v);
    }
}

// x blocks cover one row's K/8 vectors; y blocks (rows, strided) fill the GPU to ~8 resident blocks per SM
dim3 grid_for(int64_t rows, int64_t K) {
    const int64_t gx = (K / 8 + 255) / 256;
    int64_t gy = (int64_t(num_sms()) * 8 + gx - 1) / gx;
    if (gy > rows) gy = rows;
    if (gy > 65535) gy = 65535;
    if (gy < 1) gy = 1;
    return dim3(unsigned(gx), unsigned(gy));
}

}  // namespace

namespace {

template <bool ROWS>
cudaError_t launch_reduce(const void* y, int y_dtype, const int32_t* ids, const float* w, int64_t T, int top_k,
                          int64_t lim, int64_t K, void* out, int out_dtype, int32_t* err_word, cudaStream_t s) {
    if (T == 0 || K == 0) return cudaSuccess;
    const dim3 g = grid_for(T, K);
#define MOE_REDUCE(YD, OD) \
    topk_reduce_kernel<YD, OD, ROWS><<<g, 256, 0, s>>>(y, ids, w, T, top_k, lim, K, out, err_word)
    if (y_dtype == MOE_BF16 && out_dtype == MOE_BF16) MOE_REDUCE(MOE_BF16, MOE_BF16);
    else if (y_dtype == MOE_BF16 && out_dtype == MOE_F32) MOE_REDUCE(MOE_BF16, MOE_F32);
    else if (y_dtype == MOE_F32 && out_dtype == MOE_BF16) MOE_REDUCE(MOE_F32, MOE_BF16);
    else MOE_REDUCE(MOE_F32, MOE_F32);
#undef MOE_REDUCE
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_topk_reduce(const void* y, int y_dtype, const int32_t* ids, const float* w, int64_t T,
                               int top_k, int E, int64_t K, void* out, int out_dtype, cudaStream_t s) {
    return launch_reduce<false>(y, y_dtype, ids, w, T, top_k, E, K, out, out_dtype, nullptr, s);
}

cudaError_t launch_rows_topk_reduce(const void* y, int y_dtype, int64_t rows, const int32_t* route_row,
                                    const float* w, int64_t T, int top_k, int64_t K, void* out, int out_dtype,
                                    int32_t* err_word, cudaStream_t s) {
    return launch_reduce<true>(y, y_dtype, route_row, w, T, top_k, rows, K, out, out_dtype, err_word, s);
}

cudaError_t launch_batched_weight(const void* y, int y_dtype, const int32_t* counts, const float* w, int E,
                                  int max_tokens, int64_t K, void* out, int out_dtype, cudaStream_t s) {
    if (E == 0 || max_tokens == 0 || K == 0) return cudaSuccess;
    const dim3 g = grid_for(int64_t(E) * max_tokens, K);
#define MOE_BW(YD, OD) batched_weight_kernel<YD, OD><<<g, 256, 0, s>>>(y, counts, w, E, max_tokens, K, out)
    if (y_dtype == MOE_BF16 && out_dtype == MOE_BF16) MOE_BW(MOE_BF16, MOE_BF16);
    else if (y_dtype == MOE_BF16 && out_dtype == MOE_F32) MOE_BW(MOE_BF16, MOE_F32);
    else if (y_dtype == MOE_F32 && out_dtype == MOE_BF16) MOE_BW(MOE_F32, MOE_BF16);
    else MOE_BW(MOE_F32, MOE_F32);
#undef MOE_BW
    return cudaGetLastError();
}

}  // namespace moe
