// bf16 grouped GEMMs on CTA pairs (tcgen05 cta_group::2) for sm_103a: the prefill regime, many tokens per
// expert.
//
// A cluster of two CTAs on two SMs issues one MMA of M = 256 weight rows x N tokens (N <= 256): each CTA
// stages 128 weight rows and N/2 token rows of every k-block in its own shared memory, and each CTA's TMEM
// holds the accumulator of its 128 weight rows for all N tokens.  Against one SM running a 128 x 256 tile,
// a k-block moves 32 KB instead of 48 KB into each SM for the same MMA work, so a 6-stage ring fits where the
// single-SM ring held 4, and the B operand is read from shared memory once for two SMs.
//
// Orientation: weights on the MMA M side and tokens on N, the swap-AB arrangement (AWS "MoE kernel
// engineering on SageMaker AI", Swap-AB: C^T = B^T A^T), so that an expert's tokens are padded to 32 only:
// 128-row token tiles padded each expert to a multiple of 128 rows, and a pair of such tiles would pad it to
// 256 (a fifth of the executed rows on the skewed prefill routing); here about 3 %.  Each weight tile is
// reused by every 256-token segment of its expert through L2 ("Cake MegaMoE EP16" FlashInfer PR 5148
// analysis, section 3: weight-tile reuse across an expert's tokens).  The tiles of experts with a single
// segment, which stream their weights for few tokens, are spread evenly among the other experts' tiles rather
// than left to run together at the end (decode_tile).
//
// Per CTA, 192 threads:
//   warp 0      TMA producer: this CTA's 128 weight rows (128-byte swizzled, through the gate/up view for
//               GEMM 1 as in the single-SM swap-AB tiles, or one contiguous 16 KB block of weights re-laid out
//               by moe_tile_weights) and its 128-row box of the tile's tokens (of which
//               the MMA reads N/2) of each k-block into a 6-stage ring; the bytes of BOTH CTAs are counted on
//               the leader CTA's "full" barrier.
//   warp 1      TMEM: allocates all 512 columns for the pair (one warp of each CTA, together).  In the
//               leader CTA (rank 0) the warp runs the MMA loop and lane 0 issues the pair's MMAs and commits
//               each stage to the "empty" barriers and each finished accumulator to the "acc_full" barriers of
//               both CTAs (multicast).
//   warps 2..9  epilogue, two warps per TMEM lane quarter taking alternate 16-token chunks: tcgen05.ld of
//               this CTA's accumulator (TMEM lane = weight row, column = token), SiLU-and-mul (GEMM 1) or
//               route weight + scatter to the (token, slot) row (GEMM 2), each 16-token block transposed
//               through the warp's own shared-memory tile into 16-byte stores; then one arrival per warp on
//               the leader's "acc_empty" barrier (16 per tile: both CTAs).
// Two 256-column accumulators let the epilogue of one tile overlap the MMAs of the next.
//
// Every mbarrier wait is bounded (2 s of globaltimer); on expiry the CTA records MOE_DEVERR_TIMEOUT and its
// roles leave their loops; both CTAs then wait (bounded) for their copies and commits in flight, meet at a
// cluster barrier and free TMEM together.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int PM = 128;                      // weight rows per CTA (the pair's MMA M = 256)
constexpr int PK = 64;                       // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int UMMA_K = 16;
constexpr int PSPAN = 256;                   // tokens per tile (MMA N; N/2 staged by each CTA)
constexpr int STAGES = 6;
constexpr int A_BYTES = PM * PK * 2;         // 16 KB of weights per CTA per k-block
constexpr int B_BYTES = (PSPAN / 2) * PK * 2;   // up to 16 KB of tokens per CTA per k-block
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SMEM = STAGES * STAGE_BYTES + 1024;
constexpr int ACC_COLS = PSPAN;              // fp32 TMEM columns per accumulator
constexpr int TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;                 // two per TMEM lane quarter, taking alternate 16-token chunks
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int EPI_TOK = PSPAN / 2;           // tokens of a tile one epilogue warp handles
constexpr uint64_t kWaitNs = 2000000000ull;
static_assert(SMEM + 13 * 1024 + 2 * EPI_WARPS * EPI_TOK * 4 + EPI_WARPS * 1024 + 4 * kMaxExperts <= 227 * 1024,
              "shared memory exceeds the opt-in limit");
static_assert(2 * ACC_COLS <= TMEM_COLS, "accumulators exceed the TMEM allocation");
static_assert(SMEM + 13 * 1024 <= 227 * 1024, "stage ring exceeds shared memory");
static_assert(STAGE_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "stage buffers must stay 1024-byte aligned");

// GEMM 2 epilogue: each epilogue warp's copy of the tile's destination rows and route weights (loaded for all
// tokens at once at the start of a tile instead of two dependent loads per token)
struct __align__(16) EpiStage {
    int32_t dst[EPI_WARPS][EPI_TOK];   // indexed by the warp's own chunks: (cb / 2) * 16 + i
    float wt[EPI_WARPS][EPI_TOK];
    // per warp, one 16-token block of its results transposed to token-major order for 16-byte stores:
    // GEMM 1 [16 tokens][16 units] bf16, GEMM 2 [16 tokens][32 columns] bf16
    uint16_t tr[EPI_WARPS][16 * 32];
};

struct __align__(8) PairCtrl {
    uint64_t full[STAGES];     // leader: both CTAs' bytes of the stage have landed
    uint64_t empty[STAGES];    // each CTA: the MMAs that read the stage completed (multicast commit)
    uint64_t acc_full[2];      // each CTA: the tile's accumulator is complete (multicast commit)
    uint64_t acc_empty[2];     // leader: the 16 epilogue warps of the pair have read the accumulator
    uint64_t drain;            // leader: every MMA issued has completed
    uint32_t tmem_base;
    volatile int abort;
};

struct PairParams {
    int gemm;            // 1 or 2
    int layout;
    int E;
    int max_tokens;
    int64_t rows_cap;
    int nkb;             // k-blocks per tile
    int nt;              // 256-row weight tiles per expert
    int w_mode;          // weights map: 0 = 3-D (k, rows, E), 1 = 5-D gate/up interleaving view,
                         // 2 = 4-D tile-contiguous (64, 128, k-blocks, E x 128-row blocks), from moe_tile_weights
    int wblocks;         // 128-row weight blocks per expert
    int64_t I, K;
    const int32_t* counts;
    const int32_t* offsets;
    const int32_t* row_route;
    const float* route_w;
    void* out;
    int out_dtype;
    int64_t out_rows;    // GEMM 2, contiguous: rows of y (routes)
    int32_t* err_word;
    int skip_first_copy; // test hook: CTA 0 never issues its first copy (timeout_test_hook)
};

MOE_DEVICE bool wait_bar(uint64_t* bar, uint32_t parity, PairCtrl& c, int32_t* err_word) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t deadline = ptx::globaltimer() + kWaitNs;
    if (ptx::mbar_wait_bounded(bar, parity, deadline, &c.abort)) return true;
    if (!c.abort) {
        c.abort = 1;
        report(err_word, MOE_DEVERR_TIMEOUT);
    }
    return false;
}

struct PTile {
    int e;
    int64_t row0;   // first token row of the tile
    int rows;       // tokens (<= PSPAN)
    int nb;         // 256-row weight tile
};

// Tile order.  An expert of one token segment streams its weights for a handful of tokens, so its tiles are
// bound by memory while the segments of a busy expert are bound by the tensor cores.  Listed expert by expert,
// the single-segment experts (the cold ones, which come last under a skewed routing) would share the last waves
// and wait on HBM together while earlier waves left it idle, so the order spreads their tiles evenly: tile slot t
// holds a single-segment tile when floor((t+1) n1 / T) > floor(t n1 / T) (n1 of the T tiles are single-segment),
// and the two kinds keep expert order among themselves, each multi-segment expert's segments together so that
// its weight tiles are reused through L2.  `single` is the inclusive prefix of single-segment tiles over experts.
// Every role of both CTAs decodes the same tile from the same table.
MOE_DEVICE PTile decode_tile(const ExpertTable& tab, const int32_t* single, int32_t n1, const PairParams& p,
                             int32_t t) {
    const int64_t T = tab.total;
    int lo = 0, hi = p.E - 1;
    int32_t local;
    if (n1 == 0 || n1 == T) {   // one kind only (e.g. every batched expert fits a segment): expert order
        lo = find_expert(tab, p.E, t);
        local = t - tiles_before(tab, lo);
    } else if (int32_t(int64_t(t + 1) * n1 / T) > int32_t(int64_t(t) * n1 / T)) {   // a single-segment tile
        const int32_t b0 = int32_t(int64_t(t) * n1 / T);
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (single[mid] > b0) hi = mid;
            else lo = mid + 1;
        }
        local = b0 - (lo > 0 ? single[lo - 1] : 0);
    } else {         // the (t - floor(t n1 / T))-th tile of the multi-segment experts
        const int32_t a = t - int32_t(int64_t(t) * n1 / T);
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (tab.tile_end[mid] - single[mid] > a) hi = mid;
            else lo = mid + 1;
        }
        local = a - (lo > 0 ? tab.tile_end[lo - 1] - single[lo - 1] : 0);
    }
    PTile tl;
    tl.e = lo;
    const int32_t seg = local / p.nt;
    tl.nb = local - seg * p.nt;
    tl.row0 = int64_t(tab.start[tl.e]) + int64_t(seg) * PSPAN;
    tl.rows = min(PSPAN, tab.count[tl.e] - seg * PSPAN);
    return tl;
}

// MMA N of a tile: its tokens rounded up to 32, so that each CTA stages a whole number of 16-row boxes.
MOE_DEVICE int pair_n(int rows) { return max(32, (rows + 31) & ~31); }

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_w,
                     const PairParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ ExpertTable tab;
    __shared__ PairCtrl ctrl;
    __shared__ EpiStage epi;
    __shared__ int32_t single[kMaxExperts];   // inclusive prefix of single-segment experts' tiles (tile order)

    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&ctrl.full[s], 1);
            ptx::mbar_init(&ctrl.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&ctrl.acc_full[b], 1);
            ptx::mbar_init(&ctrl.acc_empty[b], 2 * EPI_WARPS);
        }
        ptx::mbar_init(&ctrl.drain, 1);
        ctrl.abort = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tm_act);
        ptx::prefetch_tmap(&tm_w);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(&ctrl.tmem_base, TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    const int nt = p.nt;
    build_expert_table(tab, p.E, p.counts, p.offsets, p.max_tokens, p.rows_cap,
                       [nt](int32_t c) { return ((c + PSPAN - 1) / PSPAN) * nt; });
    if (warp == 2) {   // one warp scans the single-segment tiles over the experts, 32 at a time
        int32_t run = 0;
        for (int e0 = 0; e0 < p.E; e0 += 32) {
            const int e = e0 + lane;
            const int32_t c = e < p.E ? tab.count[e] : 0;
            int32_t v = (c > 0 && c <= PSPAN) ? nt : 0;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int32_t n = __shfl_up_sync(0xffffffffu, v, d);
                if (lane >= d) v += n;
            }
            if (e < p.E) single[e] = run + v;
            run += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();     // barriers initialised and TMEM allocated in both CTAs before any cross-CTA use
    ptx::tc_fence_after();
    const uint32_t tmem_base = ctrl.tmem_base;
    // the pair's allocation is collective, so both CTAs must hold the same TMEM address
    const uint32_t peer_tmem = ptx::ld_shared_cluster_u32(ptx::map_to_rank(ptx::smem_addr(&ctrl.tmem_base), rank ^ 1));
    const bool pair_ok = peer_tmem == tmem_base;
    if (!pair_ok && threadIdx.x == 0) report(p.err_word, MOE_DEVERR_INTERNAL);
    const int32_t total = pair_ok ? tab.total : 0;
    const int32_t cid = int32_t(ptx::cluster_id_x()), ncl = int32_t(ptx::cluster_count_x());
    const int32_t n1 = p.E > 0 ? single[p.E - 1] : 0;   // single-segment tiles in all

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            // weights are reused by every token segment of their expert (L2), tokens by every weight tile
            const uint64_t pol = ptx::policy_evict_last();
            uint32_t it = 0;
            for (int32_t t = cid; t < total && !ctrl.abort; t += ncl) {
                const PTile tl = decode_tile(tab, single, n1, p, t);
                const int n = pair_n(tl.rows);
                // one 128-row token box per CTA (rows past the tile are never read by the MMA; past the end of
                // the activations the box is zero-filled): 2 copies per stage and CTA, a constant byte count
                const uint32_t bytes = 2u * uint32_t(STAGE_BYTES);   // both CTAs
                const int wblk = 2 * tl.nb + int(rank);              // this CTA's 128-row weight block
                const int64_t trow = tl.row0 + int64_t(rank) * (n / 2);
                bool ok = true;
                for (int kb = 0; kb < p.nkb; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!wait_bar(&ctrl.empty[s], ph ^ 1, ctrl, p.err_word)) { ok = false; break; }
                    if (leader) ptx::mbar_arrive_expect_tx(&ctrl.full[s], bytes);
                    if (p.skip_first_copy && blockIdx.x == 0 && it == 0) continue;   // bytes that never arrive
                    const uint32_t fb = ptx::map_to_rank(ptx::smem_addr(&ctrl.full[s]), 0);
                    uint8_t* sa = smem + s * STAGE_BYTES;
                    uint8_t* sb = sa + A_BYTES;
                    const int k0 = kb * PK;
                    if (p.w_mode == 1)
                        ptx::tma_load_5d_pair(sa, &tm_w, fb, k0, 0, 0, wblk * (PM / 32), tl.e, pol);
                    else if (p.w_mode == 2)   // one contiguous 16 KB block per k-block
                        ptx::tma_load_4d_pair(sa, &tm_w, fb, 0, 0, kb, tl.e * p.wblocks + wblk, pol);
                    else
                        ptx::tma_load_3d_pair(sa, &tm_w, fb, k0, wblk * PM, tl.e, pol);
                    ptx::tma_load_2d_pair(sb, &tm_act, fb, k0, int32_t(trow), pol);
                }
                if (!ok) break;
            }
            // copies in flight land and the commits of every stage issued arrive before the CTA can leave
            // (the leader's full barriers count both CTAs' bytes); one bounded deadline for all of it
            const uint64_t deadline = ptx::globaltimer() + kWaitNs / 4;
            volatile int never = 0;
            for (uint32_t j = it > STAGES ? it - STAGES : 0; j < it; ++j) {
                if (leader) ptx::mbar_wait_bounded(&ctrl.full[j % STAGES], (j / STAGES) & 1, deadline, &never);
                ptx::mbar_wait_bounded(&ctrl.empty[j % STAGES], (j / STAGES) & 1, deadline, &never);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader CTA only)
        // the whole warp runs the loop (waits, addresses and descriptors are warp-uniform) and lane 0 issues
        // every MMA and commit
        if (leader) {
            const uint32_t issue = lane == 0;
            uint32_t it = 0, tc = 0;
            for (int32_t t = cid; t < total && !ctrl.abort; t += ncl, ++tc) {
                const PTile tl = decode_tile(tab, single, n1, p, t);
                const int buf = int(tc & 1);
                const uint32_t aph = (tc >> 1) & 1;
                if (!__all_sync(0xffffffffu, wait_bar(&ctrl.acc_empty[buf], aph ^ 1, ctrl, p.err_word))) break;
                ptx::tc_fence_after();
                const uint32_t idesc = ptx::idesc_bf16(2 * PM, pair_n(tl.rows));
                const uint32_t d_tmem = tmem_base + uint32_t(buf * ACC_COLS);
                bool ok = true;
                for (int kb = 0; kb < p.nkb; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!__all_sync(0xffffffffu, wait_bar(&ctrl.full[s], ph, ctrl, p.err_word))) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_addr(smem + s * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < PK / UMMA_K; ++kk)
                        ptx::mma_f16_pair_by(issue, d_tmem, ptx::smem_desc_sw128(sa + kk * UMMA_K * 2),
                                             ptx::smem_desc_sw128(sb + kk * UMMA_K * 2), idesc, (kb | kk) != 0);
                    ptx::mma_commit_pair_by(issue, &ctrl.empty[s], 0x3);
                }
                if (!ok) break;
                ptx::mma_commit_pair_by(issue, &ctrl.acc_full[buf], 0x3);
            }
            // all MMAs issued (and the commits before this one) complete before TMEM is released
            ptx::mma_commit_pair_by(issue, &ctrl.drain, 0x1);
            const uint64_t deadline = ptx::globaltimer() + kWaitNs / 4;
            volatile int never = 0;
            ptx::mbar_wait_bounded(&ctrl.drain, 0, deadline, &never);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;                       // TMEM lane quarter of this warp
        const int sub = (warp - 2) >> 2;              // chunks cb with cb % 2 == sub
        const uint32_t lane_base = uint32_t(q * 32) << 16;
        uint32_t tc = 0;
        for (int32_t t = cid; t < total; t += ncl, ++tc) {
            const PTile tl = decode_tile(tab, single, n1, p, t);
            const int buf = int(tc & 1);
            const uint32_t aph = (tc >> 1) & 1;
            if (!wait_bar(&ctrl.acc_full[buf], aph, ctrl, p.err_word)) break;
            ptx::tc_fence_after();
            const uint32_t tacc = tmem_base + lane_base + uint32_t(buf * ACC_COLS);
            const int wblk = 2 * tl.nb + int(rank);
            const int n_tok = tl.rows;
            const int n_chunks = (n_tok + 15) / 16;
            if (p.gemm == 1) {
                // lane l < 16 holds the gate, lane l + 16 the up value of unit u = 64*wblk + 16*q + (l & 15) for
                // 16 tokens of a chunk.  Lane l computes the even tokens' h of its unit and lane l + 16 the odd
                // ones: each sends the partner the value it lacks (one exchange per token pair), so every SiLU
                // runs on a full warp.  The 16 x 16 block of h goes through this warp's shared-memory tile to
                // token-major order and leaves as one 16-byte store per lane (two lanes per token row).
                const int64_t unit0 = int64_t(wblk) * 64 + q * 16;
                uint16_t* h = static_cast<uint16_t*>(p.out);
                uint16_t* tr = epi.tr[warp - 2];
                const bool up_lane = lane >= 16;
                const int u_local = lane & 15;
                uint32_t va[16], vb[16];
                if (sub < n_chunks) ptx::tmem_ld_32x32b_x16(tacc + sub * 16, va);
#pragma unroll 1
                for (int cb = sub; cb < n_chunks; cb += 2) {
                    ptx::tmem_ld_wait_regs16(va);
#pragma unroll
                    for (int i = 0; i < 16; ++i) vb[i] = va[i];
                    if (cb + 2 < n_chunks) ptx::tmem_ld_32x32b_x16(tacc + (cb + 2) * 16, va);
                    __syncwarp();                                  // the previous block has been read back
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float even = __uint_as_float(vb[2 * j]), odd = __uint_as_float(vb[2 * j + 1]);
                        const float recv = __shfl_xor_sync(0xffffffffu, up_lane ? even : odd, 16);
                        const float g = up_lane ? recv : even;     // gate of token 2j (+1 for up lanes)
                        const float u = up_lane ? odd : recv;      // up of the same token
                        tr[(2 * j + (up_lane ? 1 : 0)) * 16 + u_local] = float_to_bf16_bits(silu_mul_fast(g, u));
                    }
                    __syncwarp();
                    const int t = lane >> 1, n = cb * 16 + t;      // token of this lane's half row
                    const uint4 v = *reinterpret_cast<const uint4*>(tr + t * 16 + (lane & 1) * 8);
                    if (n < n_tok)
                        *reinterpret_cast<uint4*>(h + (tl.row0 + n) * p.I + unit0 + (lane & 1) * 8) = v;
                }
            } else {
                const int64_t col = int64_t(wblk) * PM + q * 32 + lane;   // output hidden index
                // destination row (-1: skip) and weight of every token of the tile, 8 per lane, loads in flight
                // together
                int32_t* dst_s = epi.dst[warp - 2];
                float* wt_s = epi.wt[warp - 2];
                __syncwarp();                                  // this warp's reads of the previous tile are done
                int32_t dr[EPI_TOK / 32];
#pragma unroll
                for (int j = 0; j < EPI_TOK / 32; ++j) {
                    // entry j*32 + lane: token (cb/2)*16 + i of chunk cb = 2*((j*32+lane)/16) + sub
                    const int e = j * 32 + lane;
                    const int n = (2 * (e >> 4) + sub) * 16 + (e & 15);
                    int32_t d = -1;
                    if (n < n_tok) {
                        const int64_t row = tl.row0 + n;
                        if (p.layout == MOE_LAYOUT_CONTIGUOUS) {
                            const int32_t route = p.row_route[row];
                            d = (route >= 0 && route < p.out_rows) ? route : -1;
                        } else {
                            d = int32_t(row);
                        }
                    }
                    dr[j] = d;
                }
#pragma unroll
                for (int j = 0; j < EPI_TOK / 32; ++j) {
                    dst_s[j * 32 + lane] = dr[j];
                    wt_s[j * 32 + lane] = (p.route_w && dr[j] >= 0) ? p.route_w[dr[j]] : 1.f;
                }
                __syncwarp();
                uint16_t* tr = epi.tr[warp - 2];
                const int64_t col0 = int64_t(wblk) * PM + q * 32;   // this warp's 32 output columns
                uint32_t va[16], vb[16];
                if (sub < n_chunks) ptx::tmem_ld_32x32b_x16(tacc + sub * 16, va);
#pragma unroll 1
                for (int cb = sub; cb < n_chunks; cb += 2) {
                    ptx::tmem_ld_wait_regs16(va);
#pragma unroll
                    for (int i = 0; i < 16; ++i) vb[i] = va[i];
                    if (cb + 2 < n_chunks) ptx::tmem_ld_32x32b_x16(tacc + (cb + 2) * 16, va);
                    const int base = (cb >> 1) * 16;               // this chunk's entries in dst_s / wt_s
                    if (p.out_dtype == MOE_BF16) {
                        // the 16 tokens x 32 columns block goes token-major through this warp's tile and leaves
                        // as two 16-byte stores per lane (two lanes per token row of 64 bytes)
                        __syncwarp();                              // the previous block has been read back
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            tr[i * 32 + lane] = float_to_bf16_bits(wt_s[base + i] * __uint_as_float(vb[i]));
                        __syncwarp();
                        // lanes 2t and 2t+1 write token t's 64 bytes as two whole 32-byte sectors: store k holds
                        // columns 16k..16k+15, 8 per lane
                        const int t = lane >> 1, h8 = (lane & 1) * 8;
                        const int32_t d = dst_s[base + t];         // -1 for skipped routes and past the tokens
                        const uint4 v0 = *reinterpret_cast<const uint4*>(tr + t * 32 + h8);
                        const uint4 v1 = *reinterpret_cast<const uint4*>(tr + t * 32 + 16 + h8);
                        if (d >= 0) {
                            uint16_t* row = static_cast<uint16_t*>(p.out) + int64_t(d) * p.K + col0;
                            *reinterpret_cast<uint4*>(row + h8) = v0;
                            *reinterpret_cast<uint4*>(row + 16 + h8) = v1;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int32_t d = dst_s[base + i];
                            if (d < 0) continue;
                            static_cast<float*>(p.out)[int64_t(d) * p.K + col] = wt_s[base + i] * __uint_as_float(vb[i]);
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader) ptx::mbar_arrive(&ctrl.acc_empty[buf]);
                else ptx::mbar_arrive_remote(ptx::map_to_rank(ptx::smem_addr(&ctrl.acc_empty[buf]), 0));
            }
        }
    }

    // both CTAs: every role is done with the other CTA's barriers and its own TMEM before the pair frees it
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// Clusters of this kernel that fit on the device at once (persistent grid), cached per device.
int pair_clusters() {
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(2 * (num_sms() / 2)));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = num_sms() / 2;
    }
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

int set_pair_smem_attr() {
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && !done[dev]) {
        if (cudaFuncSetAttribute(gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) != cudaSuccess)
            return fail(MOE_ERR_LAUNCH, "cudaFuncSetAttribute(max dynamic smem) failed for the CTA-pair GEMM");
        done[dev] = true;
    }
    return MOE_OK;
}

}  // namespace

int launch_gemm_pair(const GemmArgs& g, cudaStream_t s) {
    if (g.a_dtype != MOE_BF16 || g.w_dtype != MOE_BF16)
        return fail(MOE_ERR_UNSUPPORTED, "CTA-pair tiles: bf16 activations and weights only");
    if (g.gemm == 1 && g.out_dtype != MOE_BF16) return fail(MOE_ERR_UNSUPPORTED, "CTA-pair GEMM 1 writes bf16 h");
    const int64_t kdim = g.gemm == 1 ? g.K : g.I;
    const int64_t wrows = g.gemm == 1 ? 2 * g.I : g.K;
    if (kdim % PK != 0) return fail(MOE_ERR_UNSUPPORTED, "CTA-pair tiles: contraction length must be a multiple of 64");
    if (wrows % (2 * PM) != 0)
        return fail(MOE_ERR_UNSUPPORTED, "CTA-pair tiles: weight rows per expert must be a multiple of 256");
    if (g.gemm == 1 && g.w1_layout == MOE_W1_GATE_UP && g.I % 16 != 0)
        return fail(MOE_ERR_UNSUPPORTED, "CTA-pair tiles: I must be a multiple of 16");
    if (g.rows_cap >= (int64_t(1) << 31)) return fail(MOE_ERR_UNSUPPORTED, "CTA-pair tiles: too many rows");
    if (g.rows_cap == 0) return MOE_OK;

    // token rows in 128-row boxes (the normal tiles' activation map) and weights in 128-row boxes (the swap-AB
    // tiles' weight map: the gate/up view for GEMM 1 on [gate; up] W1)
    const int w_mode = g.w1_layout == MOE_W_TILED ? 2 : ((g.gemm == 1 && g.w1_layout == MOE_W1_GATE_UP) ? 1 : 0);
    MapSet m_tok, m_w;
    int rc = cached_maps(g, TC_NORMAL, false, kdim, wrows, w_mode, &m_tok);
    if (rc) return rc;
    rc = cached_maps(g, TC_SWAP, false, kdim, wrows, w_mode, &m_w);
    if (rc) return rc;

    PairParams p{};
    p.gemm = g.gemm;
    p.layout = g.layout;
    p.E = g.E;
    p.max_tokens = g.max_tokens;
    p.rows_cap = g.rows_cap;
    p.nkb = int(kdim / PK);
    p.nt = int(wrows / (2 * PM));
    p.w_mode = w_mode;
    p.wblocks = int(wrows / PM);
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
    p.skip_first_copy = timeout_test_hook() ? 1 : 0;

    rc = set_pair_smem_attr();
    if (rc) return rc;
    // upper bound on the tiles, then as many clusters as are resident at once (persistent)
    int64_t segs;
    if (g.layout == MOE_LAYOUT_CONTIGUOUS) segs = (g.rows_cap + PSPAN - 1) / PSPAN + g.E;
    else segs = int64_t(g.E) * ((g.max_tokens + PSPAN - 1) / PSPAN);
    const int64_t tiles = segs * p.nt;
    if (tiles == 0) return MOE_OK;
    const int clusters = int(std::min<int64_t>(tiles, pair_clusters()));
    gemm_pair_kernel<<<2 * clusters, THREADS, SMEM, s>>>(m_tok.act, m_w.w, p);
    return check_launch("gemm_pair_kernel");
}

}  // namespace moe
