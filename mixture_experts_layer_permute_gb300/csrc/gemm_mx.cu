// Block-scaled MXFP8 grouped GEMMs for sm_103a: E4M3 activations x E4M3
// weights, one E8M0 scale per 32 along the contraction on both operands,
// fp32 accumulate in TMEM (tcgen05.mma kind::mxf8f6f4, scale_vec::1X).  The
// activations are quantised on the fly by mxfp8_quantize_block32 ("Fused MoE
// Modular Kernel", prepare(): input activation quantisation; apply():
// quantisation of the intermediate between act+mul and W2); the weights are
// stored quantised ("Cake MegaMoE EP16" FlashInfer PR 5148 analysis, section 2).
//
// Swap-AB tiles only (AWS "MoE kernel engineering on SageMaker AI", Swap-AB):
// 128 weight rows on the MMA M side, up to 64 of an expert's tokens on N, so a
// weight tile is streamed once for all of them.  Persistent, one CTA per SM:
//   warp 0      TMA producer: per 128-wide k slice, the weight codes (128 rows
//               x 128 B) and the token codes (16-row boxes) into an 8-stage
//               ring, 128-byte swizzled.  Weights carry an L2 evict-first hint.
//   warp 1      MMA issuer: four K=32 MMAs per slice (scale-factor ids 0..3)
//               into one of two 64-column TMEM accumulators.
//   warps 2..5  epilogue: tcgen05.ld, SiLU-and-mul (GEMM 1) or route weight +
//               scatter to the (token, slot) row (GEMM 2).
//   warps 6..21 scale writers, four groups of four warps taking slices in turn:
//               each thread loads one 32-bit word (the 4 scales of the slice)
//               for 4 weight rows and 2 token rows and writes them into the
//               slice's scale slot in TMEM with tcgen05.st.
// Scale factors in TMEM, as the MMA reads them (M = 128, N <= 128; measured on
// the hardware against other placements): the scales of operand row r lie in
// lane r % 32 of each of the four lane quarters, 32-bit column r / 32, and the
// byte of that word is the k block within the slice (the MMA's scale-factor
// id).  Each warp may only write its own lane quarter, so all four warps of a
// group write the same words.
//
// Every mbarrier wait is bounded (2 s of globaltimer); on expiry the kernel
// records MOE_DEVERR_TIMEOUT, lets its copies in flight land, frees TMEM and
// returns.
#include <cuda.h>

#include <mutex>
#include <string>
#include <unordered_map>

#include "common.cuh"
#include "internal.h"
#include "mx_codec.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int BM = 128;                      // weight rows per tile (MMA M)
constexpr int KS = 128;                      // contraction per slice: 128 codes = one swizzle row
constexpr int MMA_K = 32;                    // E4M3 k per MMA
constexpr int SPAN = 64;                     // tokens per tile (MMA N = 64)
constexpr int TOK_BOX = 16;                  // token rows per TMA box
constexpr int STAGES = 8;
constexpr int A_BYTES = BM * KS;             // 16 KB of weight codes per slice
constexpr int B_BYTES = SPAN * KS;           // 8 KB of token codes per slice
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SMEM = STAGES * STAGE_BYTES + 1024;
constexpr int ACC_COLS = SPAN;               // TMEM columns per accumulator
constexpr int SF_COL = 2 * ACC_COLS;         // first scale slot column
constexpr int SF_SLOT = 16;                  // columns per slot: A scales 0..3, B scales 8..11
constexpr int SF_B = 8;                      // B scales' offset in a slot (both start 8-column aligned)
constexpr int TMEM_COLS = 256;
constexpr int SF_GROUPS = 4;                 // scale-writer groups of 4 warps
constexpr int THREADS = 192 + SF_GROUPS * 128;
constexpr uint32_t SF_ONE = 0x7F7F7F7Fu;     // four scales of 2^0
constexpr uint64_t kWaitNs = 2000000000ull;
static_assert(SF_COL + STAGES * SF_SLOT <= TMEM_COLS, "scale slots exceed the TMEM allocation");
static_assert(SMEM + 14 * 1024 <= 227 * 1024, "stage ring exceeds shared memory");

struct __align__(8) Ctrl {
    uint64_t full[STAGES];      // TMA bytes of the slice landed
    uint64_t empty[STAGES];     // MMA done with the slice (smem and scale slot)
    uint64_t sf_full[STAGES];   // scale slot written (4 warps)
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint64_t xq[2];             // fused h quantisation: block maxima of a warp pair exchanged (2 warps)
    float xmax[2][2][2][16];    // [warp pair][chunk parity][warp of the pair][token of the chunk]
    uint32_t tmem_base;
    volatile int abort;
};

struct MxParams {
    int gemm;            // 1 or 2
    int layout;
    int E;
    int max_tokens;
    int64_t rows_cap;
    int nks;             // k slices per tile
    int nt;              // weight blocks (128 rows) per expert
    int w_mode;          // weights map: 0 = 3-D (k, rows, E), 1 = 5-D gate/up interleaving view,
                         // 2 = 4-D tile-contiguous codes (128, 128, slices, E x 128-row blocks)
    int64_t I, K;
    const int32_t* counts;
    const int32_t* offsets;
    const int32_t* row_route;
    const float* route_w;
    void* out;
    int out_dtype;
    int64_t out_rows;
    int32_t* err_word;
    const uint8_t* a_scale;   // (rows_cap, kdim/32)
    const uint8_t* w_scale;   // (E, wrows, kdim/32)
    int64_t wrows;
    int64_t nsb;              // scale bytes per row (kdim / 32)
    uint8_t* h_scale;         // GEMM 1 with E4M3 h: E8M0 scales (rows_cap, I/32); NULL: bf16 h
    int skip_first_copy;      // test hook: CTA 0 never issues its first copy (timeout_test_hook, gemm_tc.cu)
};

MOE_DEVICE bool wait_bar(uint64_t* bar, uint32_t parity, Ctrl& c, int32_t* err_word) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t deadline = ptx::globaltimer() + kWaitNs;
    if (ptx::mbar_wait_bounded(bar, parity, deadline, &c.abort)) return true;
    if (!c.abort) {
        c.abort = 1;
        report(err_word, MOE_DEVERR_TIMEOUT);
    }
    return false;
}

struct Tile {
    int e;
    int64_t row0;   // first token row
    int rows;       // tokens (<= SPAN)
    int nb;         // weight block
};

MOE_DEVICE Tile decode_tile(const ExpertTable& tab, const MxParams& p, int32_t t) {
    Tile tl;
    tl.e = find_expert(tab, p.E, t);
    const int32_t local = t - tiles_before(tab, tl.e);
    const int32_t seg = local / p.nt;
    tl.nb = local - seg * p.nt;
    tl.row0 = int64_t(tab.start[tl.e]) + int64_t(seg) * SPAN;
    tl.rows = min(SPAN, tab.count[tl.e] - seg * SPAN);
    return tl;
}

// Weight row (within the expert) held by row r of weight block nb, in the order the weight map delivers it.
MOE_DEVICE int64_t tile_weight_row(const MxParams& p, int nb, int r) {
    if (p.w_mode == 1) {   // [gate; up] rows seen through the interleave-16 view
        const int64_t unit = int64_t(nb) * 64 + (r >> 5) * 16 + (r & 15);
        return ((r >> 4) & 1) * p.I + unit;
    }
    return int64_t(nb) * BM + r;
}

__global__ void __launch_bounds__(THREADS, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_w,
                   const MxParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ ExpertTable tab;
    __shared__ Ctrl ctrl;

    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&ctrl.full[s], 1);
            ptx::mbar_init(&ctrl.empty[s], 1);
            ptx::mbar_init(&ctrl.sf_full[s], 4);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&ctrl.acc_full[b], 1);
            ptx::mbar_init(&ctrl.acc_empty[b], 4);
        }
        ptx::mbar_init(&ctrl.drain, 1);
        ptx::mbar_init(&ctrl.xq[0], 2);
        ptx::mbar_init(&ctrl.xq[1], 2);
        ctrl.abort = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tm_act);
        ptx::prefetch_tmap(&tm_w);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&ctrl.tmem_base, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    const int nt = p.nt;
    build_expert_table(tab, p.E, p.counts, p.offsets, p.max_tokens, p.rows_cap,
                       [nt](int32_t c) { return ((c + SPAN - 1) / SPAN) * nt; });
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = ctrl.tmem_base;
    const int32_t total = tab.total;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_stream = ptx::policy_evict_first();
            const uint64_t pol_keep = ptx::policy_evict_last();
            uint32_t it = 0;
            for (int32_t t = blockIdx.x; t < total && !ctrl.abort; t += gridDim.x) {
                const Tile tl = decode_tile(tab, p, t);
                const int nbox = (tl.rows + TOK_BOX - 1) / TOK_BOX;
                const uint32_t bytes = uint32_t(A_BYTES + nbox * TOK_BOX * KS);
                bool ok = true;
                for (int kb = 0; kb < p.nks; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!wait_bar(&ctrl.empty[s], ph ^ 1, ctrl, p.err_word)) { ok = false; break; }
                    uint8_t* sa = smem + s * STAGE_BYTES;
                    uint8_t* sb = sa + A_BYTES;
                    ptx::mbar_arrive_expect_tx(&ctrl.full[s], bytes);
                    if (p.skip_first_copy && blockIdx.x == 0 && it == 0) continue;   // bytes that never arrive
                    const int k0 = kb * KS;
                    const int row_w = tl.nb * BM;
                    if (p.w_mode == 1)
                        ptx::tma_load_5d(sa, &tm_w, &ctrl.full[s], k0, 0, 0, row_w / 32, tl.e, pol_stream);
                    else if (p.w_mode == 2)   // one contiguous 16 KB block per slice
                        ptx::tma_load_4d(sa, &tm_w, &ctrl.full[s], 0, 0, kb, tl.e * p.nt + tl.nb, pol_stream);
                    else
                        ptx::tma_load_3d(sa, &tm_w, &ctrl.full[s], k0, row_w, tl.e, pol_stream);
                    for (int b = 0; b < nbox; ++b)
                        ptx::tma_load_2d(sb + b * TOK_BOX * KS, &tm_act, &ctrl.full[s], k0,
                                         int32_t(tl.row0 + b * TOK_BOX), pol_keep);
                }
                if (!ok) break;
            }
            // every copy issued so far lands before the CTA can exit (bounded)
            for (uint32_t j = it > STAGES ? it - STAGES : 0; j < it; ++j) {
                const uint64_t deadline = ptx::globaltimer() + kWaitNs / 4;
                volatile int never = 0;
                ptx::mbar_wait_bounded(&ctrl.full[j % STAGES], (j / STAGES) & 1, deadline, &never);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc0 = ptx::idesc_mxf8(BM, SPAN);
            uint32_t it = 0, tc = 0;
            for (int32_t t = blockIdx.x; t < total && !ctrl.abort; t += gridDim.x, ++tc) {
                const int buf = tc & 1;
                const uint32_t aph = (tc >> 1) & 1;
                if (!wait_bar(&ctrl.acc_empty[buf], aph ^ 1, ctrl, p.err_word)) break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + uint32_t(buf * ACC_COLS);
                bool ok = true;
                for (int kb = 0; kb < p.nks; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!wait_bar(&ctrl.full[s], ph, ctrl, p.err_word)) { ok = false; break; }
                    if (!wait_bar(&ctrl.sf_full[s], ph, ctrl, p.err_word)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_addr(smem + s * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    const uint32_t sf = tmem_base + uint32_t(SF_COL + s * SF_SLOT);
#pragma unroll
                    for (int kk = 0; kk < KS / MMA_K; ++kk) {
                        const uint64_t ad = ptx::smem_desc_sw128(sa + kk * MMA_K);
                        const uint64_t bd = ptx::smem_desc_sw128(sb + kk * MMA_K);
                        ptx::mma_mxf8(d_tmem, ad, bd, idesc0 | ptx::idesc_sf_ids(kk, kk), sf, sf + SF_B,
                                      (kb | kk) != 0);
                    }
                    ptx::mma_commit(&ctrl.empty[s]);
                }
                if (!ok) break;
                ptx::mma_commit(&ctrl.acc_full[buf]);
            }
            // all MMAs issued by this thread complete before TMEM is released
            ptx::mma_commit(&ctrl.drain);
            const uint64_t deadline = ptx::globaltimer() + kWaitNs / 4;
            volatile int never = 0;
            ptx::mbar_wait_bounded(&ctrl.drain, 0, deadline, &never);
        }
        __syncwarp();
    } else if (warp >= 6) {
        // ------------------------------------------------------------ scale writers
        const int grp = (warp - 6) >> 2;
        const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
        uint32_t it = 0;
        for (int32_t t = blockIdx.x; t < total && !ctrl.abort; t += gridDim.x) {
            const Tile tl = decode_tile(tab, p, t);
            // this lane's rows: weight rows 32c + lane (c < 4) and tokens lane, 32 + lane of the tile
            const uint8_t* wrow[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                wrow[c] = p.w_scale + (int64_t(tl.e) * p.wrows + tile_weight_row(p, tl.nb, 32 * c + lane)) * p.nsb;
            const uint8_t* trow0 = lane < tl.rows ? p.a_scale + (tl.row0 + lane) * p.nsb : nullptr;
            const uint8_t* trow1 = lane + 32 < tl.rows ? p.a_scale + (tl.row0 + 32 + lane) * p.nsb : nullptr;
            bool ok = true;
            for (int kb = 0; kb < p.nks; ++kb, ++it) {
                if (int(it % SF_GROUPS) != grp) continue;   // another group's slice
                uint32_t wa[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) wa[c] = __ldg(reinterpret_cast<const uint32_t*>(wrow[c] + 4 * kb));
                const uint32_t tb0 = trow0 ? __ldg(reinterpret_cast<const uint32_t*>(trow0 + 4 * kb)) : SF_ONE;
                const uint32_t tb1 = trow1 ? __ldg(reinterpret_cast<const uint32_t*>(trow1 + 4 * kb)) : SF_ONE;
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1;
                if (!wait_bar(&ctrl.empty[s], ph ^ 1, ctrl, p.err_word)) { ok = false; break; }
                ptx::tc_fence_after();   // the MMAs that last read this slot have completed
                const uint32_t sf = tmem_base + lane_base + uint32_t(SF_COL + s * SF_SLOT);
                ptx::tmem_st_32x32b_x4(sf, wa[0], wa[1], wa[2], wa[3]);
                ptx::tmem_st_32x32b_x4(sf + SF_B, tb0, tb1, SF_ONE, SF_ONE);
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&ctrl.sf_full[s]);
            }
            if (!ok) break;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                       // TMEM lane quarter of this warp
        const uint32_t lane_base = uint32_t(q * 32) << 16;
        uint32_t tc = 0;
        uint32_t xc = 0;                              // fused h quantisation: chunks exchanged so far
        for (int32_t t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            const Tile tl = decode_tile(tab, p, t);
            const int buf = tc & 1;
            const uint32_t aph = (tc >> 1) & 1;
            if (!wait_bar(&ctrl.acc_full[buf], aph, ctrl, p.err_word)) break;
            ptx::tc_fence_after();
            const uint32_t tacc = tmem_base + lane_base + uint32_t(buf * ACC_COLS);
            // TMEM lane = weight row of the tile, column = token
            const int n_tok = tl.rows;
            const int n_chunks = (n_tok + 15) / 16;
            if (p.gemm == 1 && p.h_scale) {
                // MXFP8 h ("Fused MoE Modular Kernel", apply(): quantisation between act+mul and W2, here in
                // the epilogue): h is rounded to bf16 as the bf16 output would be, a block of 32 units along I
                // is held by two warps (16 units each: q = 2j, 2j + 1), which exchange their block maxima
                // through shared memory, then each lane writes its unit's code and lane 0 of the even warp the
                // scale -- the same codes mxfp8_quantize_block32 makes from the bf16 h.
                const int64_t unit = int64_t(tl.nb) * 64 + q * 16 + (lane & 15);
                const int pair = q >> 1, half = q & 1;
                uint8_t* hc = static_cast<uint8_t*>(p.out);
                bool ok = true;
#pragma unroll 1
                for (int cb = 0; cb < n_chunks; ++cb, ++xc) {
                    uint32_t v[16];
                    ptx::tmem_ld_32x32b_x16(tacc + cb * 16, v);
                    ptx::tmem_ld_wait();
                    float hv[16], mx[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float mine = __uint_as_float(v[i]);
                        const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
                        const float g = lane < 16 ? mine : other;
                        const float u = lane < 16 ? other : mine;
                        hv[i] = bf16_bits_to_float(float_to_bf16_bits(silu_mul(g, u)));
                        float m = fabsf(hv[i]);
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                        mx[i] = m;   // max over this warp's 16 units (both lane halves hold the same)
                    }
                    const int par = xc & 1;
                    float* mine_buf = ctrl.xmax[pair][par][half];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (lane == i) mine_buf[i] = mx[i];
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&ctrl.xq[pair]);
                    if (!wait_bar(&ctrl.xq[pair], xc & 1, ctrl, p.err_word)) { ok = false; break; }
                    const float* other_buf = ctrl.xmax[pair][par][half ^ 1];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int n = cb * 16 + i;
                        const float bm = fmaxf(mx[i], other_buf[i]);
                        const int code = mx_scale_code(bm);
                        const uint8_t c = uint8_t(mx_cvt_e4m3x2(hv[i] * mx_inv_scale(code), 0.f) & 0xFFu);
                        if (n < n_tok) {
                            if (lane < 16) hc[(tl.row0 + n) * p.I + unit] = c;
                            if (half == 0 && lane == 0)
                                p.h_scale[(tl.row0 + n) * (p.I / 32) + int64_t(tl.nb) * 2 + pair] = uint8_t(code);
                        }
                    }
                }
                if (!ok) break;
            } else if (p.gemm == 1) {
                // lanes 0..15: gate of unit u, lanes 16..31: up of unit u, u = 64*nb + 16*q + (lane & 15)
                const int64_t unit = int64_t(tl.nb) * 64 + q * 16 + (lane & 15);
                uint16_t* h = static_cast<uint16_t*>(p.out);
#pragma unroll 1
                for (int cb = 0; cb < n_chunks; ++cb) {
                    uint32_t v[16];
                    ptx::tmem_ld_32x32b_x16(tacc + cb * 16, v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float mine = __uint_as_float(v[i]);
                        const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
                        const float g = lane < 16 ? mine : other;
                        const float u = lane < 16 ? other : mine;
                        const int n = cb * 16 + i;
                        // lanes 0..15 store even tokens, 16..31 odd tokens of each pair
                        if (((i & 1) == (lane >> 4)) && n < n_tok)
                            h[(tl.row0 + n) * p.I + unit] = float_to_bf16_bits(silu_mul(g, u));
                    }
                }
            } else {
                const int64_t col = int64_t(tl.nb) * BM + q * 32 + lane;   // output hidden index
#pragma unroll 1
                for (int cb = 0; cb < n_chunks; ++cb) {
                    uint32_t v[16];
                    ptx::tmem_ld_32x32b_x16(tacc + cb * 16, v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int n = cb * 16 + i;
                        if (n >= n_tok) break;
                        const int64_t row = tl.row0 + n;
                        int64_t dst_row;
                        float wt = 1.f;
                        if (p.layout == MOE_LAYOUT_CONTIGUOUS) {
                            const int32_t route = p.row_route[row];
                            if (route < 0 || route >= p.out_rows) continue;
                            dst_row = route;
                            if (p.route_w) wt = p.route_w[route];
                        } else {
                            dst_row = row;
                            if (p.route_w) wt = p.route_w[row];
                        }
                        const float val = wt * __uint_as_float(v[i]);
                        if (p.out_dtype == MOE_BF16)
                            static_cast<uint16_t*>(p.out)[dst_row * p.K + col] = float_to_bf16_bits(val);
                        else
                            static_cast<float*>(p.out)[dst_row * p.K + col] = val;
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&ctrl.acc_empty[buf]);
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem_base, TMEM_COLS);
}

// ---- host ----------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Byte tensor map, 128-byte swizzle (every box here is 128 bytes wide).
int make_byte_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                  const cuuint32_t* box, const char* what) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(MOE_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, cuuint32_t(rank), const_cast<void*>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(MOE_ERR_ALIGNMENT, std::string("cuTensorMapEncodeTiled failed for ") + what + " (CUresult " +
                                           std::to_string(int(r)) + ")");
    return MOE_OK;
}

struct MapKey {
    int dev;
    const void* a;
    const void* w;
    int64_t kdim, rows_cap, wrows, I, K;
    int E, gemm, w_mode;
    bool operator==(const MapKey& o) const {
        return dev == o.dev && a == o.a && w == o.w && kdim == o.kdim && rows_cap == o.rows_cap &&
               wrows == o.wrows && I == o.I && K == o.K && E == o.E && gemm == o.gemm && w_mode == o.w_mode;
    }
};

struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        size_t h = std::hash<const void*>()(k.a) * 31 + std::hash<const void*>()(k.w);
        h = h * 31 + std::hash<int64_t>()(k.kdim * 1000003 + k.rows_cap);
        h = h * 31 + std::hash<int64_t>()(k.wrows * 7 + k.I * 13 + k.K * 17 + k.E);
        return h * 31 + size_t(k.gemm * 4 + k.w_mode + k.dev * 64);
    }
};

struct MapPair {
    CUtensorMap act, w;
};

std::mutex g_mu;
std::unordered_map<MapKey, MapPair, MapKeyHash> g_maps;

int build_maps(const GemmArgs& g, int64_t kdim, int64_t wrows, int w_mode, MapPair* mp) {
    {
        cuuint64_t dims[2] = {cuuint64_t(kdim), cuuint64_t(g.rows_cap)};
        cuuint64_t str[1] = {cuuint64_t(kdim)};
        cuuint32_t box[2] = {KS, TOK_BOX};
        int rc = make_byte_map(&mp->act, g.a, 2, dims, str, box, "MXFP8 activation codes");
        if (rc) return rc;
    }
    if (w_mode == 2) {
        // tile-contiguous codes (moe_tile_weights): [E x 128-row blocks][slices][128 rows][128 codes]
        cuuint64_t dims[4] = {cuuint64_t(KS), 128, cuuint64_t(kdim / KS), cuuint64_t(g.E * (wrows / 128))};
        cuuint64_t str[3] = {cuuint64_t(KS), cuuint64_t(128 * KS), cuuint64_t(kdim / KS * 128 * KS)};
        cuuint32_t box[4] = {KS, 128, 1, 1};
        return make_byte_map(&mp->w, g.w, 4, dims, str, box, g.gemm == 1 ? "W1 codes (tiled)" : "W2 codes (tiled)");
    }
    if (w_mode == 1) {
        // W1[e] (2I, K) seen as (K, 16, 2, I/16): row = half*I + 16*blk + q
        cuuint64_t dims[5] = {cuuint64_t(g.K), 16, 2, cuuint64_t(g.I / 16), cuuint64_t(g.E)};
        cuuint64_t str[4] = {cuuint64_t(g.K), cuuint64_t(g.I * g.K), cuuint64_t(16 * g.K), cuuint64_t(2 * g.I * g.K)};
        cuuint32_t box[5] = {KS, 16, 2, BM / 32, 1};
        return make_byte_map(&mp->w, g.w, 5, dims, str, box, "W1 codes (gate/up view)");
    }
    cuuint64_t dims[3] = {cuuint64_t(kdim), cuuint64_t(wrows), cuuint64_t(g.E)};
    cuuint64_t str[2] = {cuuint64_t(kdim), cuuint64_t(wrows * kdim)};
    cuuint32_t box[3] = {KS, BM, 1};
    return make_byte_map(&mp->w, g.w, 3, dims, str, box, g.gemm == 1 ? "W1 codes" : "W2 codes");
}

int set_smem_attr() {
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && !done[dev]) {
        if (cudaFuncSetAttribute(gemm_mx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) != cudaSuccess)
            return fail(MOE_ERR_LAUNCH, "cudaFuncSetAttribute(max dynamic smem) failed");
        done[dev] = true;
    }
    return MOE_OK;
}

}  // namespace

int launch_gemm_mx(const GemmArgs& g, cudaStream_t s) {
    if (g.a_dtype != MOE_E4M3 || g.w_dtype != MOE_E4M3)
        return fail(MOE_ERR_UNSUPPORTED, "block-scaled MXFP8 path: E4M3 activations and weights only");
    if (!g.a_scale || !g.w_scale) return fail(MOE_ERR_INVALID_ARG, "block-scaled MXFP8 path: scales missing");
    if (g.gemm == 1 && g.out_dtype != MOE_BF16 && g.out_dtype != MOE_E4M3)
        return fail(MOE_ERR_UNSUPPORTED, "MXFP8 GEMM 1 writes bf16 or MXFP8 h");
    if (g.gemm == 1 && g.out_dtype == MOE_E4M3 && !g.out_scale)
        return fail(MOE_ERR_INVALID_ARG, "MXFP8 h needs its scale output");
    const int64_t kdim = g.gemm == 1 ? g.K : g.I;
    if (kdim % KS != 0)
        return fail(MOE_ERR_UNSUPPORTED, "block-scaled MXFP8 path: contraction length must be a multiple of 128");
    const int64_t wrows = g.gemm == 1 ? 2 * g.I : g.K;
    if (wrows % BM != 0)
        return fail(MOE_ERR_UNSUPPORTED, "block-scaled MXFP8 path: weight rows per expert must be a multiple of 128");
    if ((reinterpret_cast<uintptr_t>(g.a_scale) & 3u) || (reinterpret_cast<uintptr_t>(g.w_scale) & 3u))
        return fail(MOE_ERR_ALIGNMENT, "block-scaled MXFP8 path: scale arrays must be 4-byte aligned");
    if (g.rows_cap >= (int64_t(1) << 31)) return fail(MOE_ERR_UNSUPPORTED, "block-scaled MXFP8 path: too many rows");
    if (g.rows_cap == 0) return MOE_OK;

    const int w_mode = g.w1_layout == MOE_W_TILED ? 2 : ((g.gemm == 1 && g.w1_layout == MOE_W1_GATE_UP) ? 1 : 0);
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    const MapKey key{dev_id, g.a, g.w, kdim, g.rows_cap, wrows, g.I, g.K, g.E, g.gemm, w_mode};
    MapPair maps;
    bool cached = false;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_maps.find(key);
        if (it != g_maps.end()) {
            maps = it->second;
            cached = true;
        }
    }
    if (!cached) {
        int rc = build_maps(g, kdim, wrows, w_mode, &maps);
        if (rc) return rc;
        std::lock_guard<std::mutex> lock(g_mu);
        if (g_maps.size() >= 256) g_maps.clear();
        g_maps[key] = maps;
    }

    MxParams p;
    p.gemm = g.gemm;
    p.layout = g.layout;
    p.E = g.E;
    p.max_tokens = g.max_tokens;
    p.rows_cap = g.rows_cap;
    p.nks = int(kdim / KS);
    p.nt = int(wrows / BM);
    p.w_mode = w_mode;
    p.I = g.I;
    p.K = g.K;
    p.counts = g.counts;
    p.offsets = g.offsets;
    p.row_route = g.row_route;
    p.route_w = g.route_w;
    p.out = g.out;
    p.out_dtype = g.out_dtype;
    p.out_rows = g.out_rows;
    p.err_word = g.err_word;
    p.a_scale = g.a_scale;
    p.w_scale = g.w_scale;
    p.wrows = wrows;
    p.nsb = kdim / 32;
    p.h_scale = (g.gemm == 1 && g.out_dtype == MOE_E4M3) ? g.out_scale : nullptr;
    p.skip_first_copy = timeout_test_hook() ? 1 : 0;

    int rc = set_smem_attr();
    if (rc) return rc;
    int64_t segs;
    if (g.layout == MOE_LAYOUT_CONTIGUOUS) segs = (g.rows_cap + SPAN - 1) / SPAN + g.E;
    else segs = int64_t(g.E) * ((g.max_tokens + SPAN - 1) / SPAN);
    const int64_t tiles = segs * p.nt;
    if (tiles == 0) return MOE_OK;
    const int grid = int(std::min<int64_t>(tiles, num_sms()));
    gemm_mx_kernel<<<grid, THREADS, SMEM, s>>>(maps.act, maps.w, p);
    return check_launch("gemm_mx_kernel");
}

}  // namespace moe
