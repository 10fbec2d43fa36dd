// moe_tile_weights: bf16 expert weights into the tile-contiguous layout the
// decode kernels stream (one 16 KB run per 128-row x 64-column block).  One
// thread moves one 16-byte vector (8 columns): writes are contiguous, reads
// are 128-byte row pieces.  An offline preparation step, run once per weight.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

__global__ void __launch_bounds__(256) tile_weights_kernel(const uint4* __restrict__ w, int which, int w1_layout,
                                                           int64_t rows, int64_t cols, int64_t total,
                                                           uint4* __restrict__ out) {
    const int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;   // output vector index
    if (v >= total) return;
    const int64_t cb_n = cols / 64, rb_n = rows / 128;
    const int j8 = int(v & 7);                 // vector within the 64-column row piece
    const int r = int((v >> 3) & 127);         // row within the block
    const int64_t blk = v >> 10;               // (e, b, c) in order, 1024 vectors per block
    const int64_t c = blk % cb_n;
    const int64_t eb = blk / cb_n;
    const int64_t b = eb % rb_n, e = eb / rb_n;
    int64_t row;
    if (which == 1 && w1_layout == MOE_W1_GATE_UP) {
        const int64_t I = rows / 2;
        const int64_t unit = 64 * b + 16 * (r >> 5) + (r & 15);
        row = ((r >> 4) & 1) ? I + unit : unit;
    } else {
        row = 128 * b + r;
    }
    out[v] = w[((e * rows + row) * cols + 64 * c) / 8 + j8];
}

}  // namespace

cudaError_t launch_tile_weights(const void* w, int which, int w1_layout, int E, int64_t rows, int64_t cols,
                                void* out, cudaStream_t s) {
    const int64_t total = int64_t(E) * rows * cols / 8;
    const int64_t blocks = (total + 255) / 256;
    tile_weights_kernel<<<unsigned(blocks), 256, 0, s>>>(static_cast<const uint4*>(w), which, w1_layout, rows, cols,
                                                          total, static_cast<uint4*>(out));
    return cudaGetLastError();
}

}  // namespace moe
