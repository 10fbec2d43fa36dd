// tcgen05 grouped GEMMs for sm_103a: persistent, warp-specialised CTAs
// (one per SM).
//
//   warp 0      TMA producer: one thread streams 64-wide k-blocks of the A and
//               B tiles into a 4-stage shared-memory ring (128-byte swizzle),
//               completing a "full" mbarrier per stage.
//   warp 1      MMA issuer: the whole warp runs the issue loop (warp-uniform
//               addresses and descriptors) and lane 0 issues tcgen05.mma
//               (kind::f16, bf16 in, fp32 accumulate) into one of two TMEM
//               accumulators and frees each stage with tcgen05.commit on its
//               "empty" mbarrier.
//   warps 2..5  epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes
//               32*(w%4)...), apply SiLU-and-mul (GEMM 1) or route weight +
//               scatter to the (token, slot) row (GEMM 2), store to global.
// The two accumulators let the epilogue of one tile overlap the MMAs of the
// next.  Tiles are listed per expert on the device (ExpertTable).
//
// Normal tiles (tokens on the MMA M side): 128 token rows x 256 weight rows.
//   GEMM 1: the 256 weight rows are 128 units as [gate16, up16] x 8, so each
//   epilogue thread holds matching gate and up columns side by side.  The
//   [gate; up] W1 layout is read through a 5-D tensor map (k, 16, 2, I/16, E)
//   that produces this order; the interleave-16 layout is read as stored.
// Swap-AB tiles (AWS "MoE kernel engineering on SageMaker AI", Swap-AB:
//   C^T = B^T A^T when tokens per expert are few): 128 weight rows on M and
//   the expert's tokens (up to 256, loaded as 16-row boxes) on N, so a weight
//   tile is read once for all of the expert's tokens.  Weight loads carry an
//   L2 evict-first hint (the weights are streamed once).
//
// MXFP8 weights (E4M3 codes + one E8M0 scale per 32 along the contraction;
//   "Cake MegaMoE EP16" FlashInfer PR 5148 analysis, section 2): swap-AB tiles
//   only, 128-wide k slices.  Two rings: TMA streams the raw codes (1 byte per
//   weight, each read once, full 128-byte lines, 128-byte swizzled) into a
//   9-stage code ring that is freed as soon as a slice is decoded; four A
//   slots hold decoded tiles in tensor memory plus the matching token tiles
//   in shared memory.  Sixteen converter warps in four groups take slices in
//   turn (group = slice index mod 4 = A slot), so four slices are in
//   conversion at once.  Once the MMA has released its slot, a group starts
//   16-byte cp.async copies of the slice's token rows into the slot (128-byte
//   swizzled, as the MMA reads them) and decodes while they land: a TMA copy
//   per slot issued by one more warp took about 0.35 us to issue under the
//   converters' load and put its latency on the slot's critical path.  Warp w
//   may only reach TMEM lanes 32*(w%4)..+31, so in its group thread (w, lane)
//   owns row 32*(w%4)+lane of the slice: 128 codes and four scales.  Decoding
//   needs no conversion instruction: the E4M3 bits placed into bf16 bit
//   positions (sign to bit 15, exponent and mantissa to bits 10..4) give
//   exactly code * 2^-120 for normal, subnormal and zero codes alike, and one
//   bf16x2 multiply by 2^(scale-7) restores the value (two multiplies when that
//   factor would leave bf16's range, scale codes above 134: a warp whose slice
//   has one takes that path for all its rows, so the common slice carries no
//   per-block test; the four factors of an ordinary scale word are formed at
//   once).  The MMA takes its A operand from TMEM.  The producer hands each
//   tile it decodes to the converters through a 4-entry shared-memory ring, so
//   that the look-up stays off their path.
//   Tokens per tile are capped at 64.  Two warps issue the MMAs, the even and
//   the odd k slices of a tile, each into its own accumulator, and the
//   epilogue adds the two: with the converter warps competing for issue slots
//   one issuing warp sustains only about one M=128, K=16 MMA per 65-120 ns
//   whatever N is (measured on GB300), which for 1-byte weights (128 x 16
//   bytes per MMA) is at or below the HBM rate; two warps double it.  When the
//   routed rows average 16 or fewer per expert, tiles hold up to 32 tokens and
//   four warps issue, two per slice parity, each half of a slice's MMAs (the
//   narrower accumulators leave TMEM room for them).  Every instruction the
//   converter and MMA warps save is an issue slot for the others, so both walk
//   only their own slices, with stage indices and parities kept incrementally.
//
// Wide tiles (bf16, batched layout): 256 token rows x 256 weight rows as two
// 128-row MMA halves that share each B stage, so an expert of up to 256 rows
// streams each weight tile once; the two halves fill TMEM, so there is one
// accumulator and 8 epilogue warps (warp w: half (w-2)/4, lane quarter w%4).
//
// Mixed tiles (bf16): one launch serves experts of 64 rows or more with
// normal 128-row tiles and smaller experts with a swap-AB tile, so a skewed
// routing does not pay a mostly empty 128-row tile per small expert.
//
// Every mbarrier wait is bounded (2 s of globaltimer); on expiry the kernel
// records MOE_DEVERR_TIMEOUT, lets its copies in flight land, frees TMEM and
// returns.
#include <cuda.h>

#include <cstdlib>
#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "internal.h"
#include "mx_codec.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int BM = 128;           // MMA M
constexpr int BK = 64;            // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int UMMA_K = 16;
constexpr int A_BYTES = BM * BK * 2;        // 16 KB
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 512;
constexpr int TOK_BOX = 16;                 // swap-AB token rows per TMA box
constexpr int MAX_STAGES = 12;
constexpr int kConvThreads = 512;           // E4M3 converter warps 6..21
constexpr uint64_t kWaitNs = 2000000000ull;

// Per variant: stage ring layout, TMEM map and CTA shape.
//   V_BF16:   smem [A 16 KB][B 32 KB] x 4 stages; TMEM: two 256-column accumulators;
//             192 threads; normal tiles, mixed launches, swap-AB tiles of up to 256 tokens
//   V_SWAP64: bf16 swap-AB tiles of up to 64 tokens: smem [A 16 KB][B 8 KB] x 8 stages (twice the
//             weight bytes in flight of V_BF16); TMEM: two 64-column accumulators; 192 threads
//   V_E4M3:   smem: 9 code stages of 128 rows x 128 B, then 4 token slots of 2 x 8 KB;
//             TMEM: two buffers of two 64-column accumulators (one per MMA issuer), then 4 bf16 A tiles
//             of 64 columns; 736 threads (+ 16 converter warps, + a second MMA warp); up to 64 tokens per
//             tile
//   V_E4M3N:  as V_E4M3 with up to 32 tokens per tile (chosen when the routed rows average 16 or fewer per
//             expert): 11 code stages, token slots of 2 x 4 KB; TMEM: two buffers of four 32-column
//             accumulators; four MMA warps (800 threads), two per slice parity, each issuing 4 of a slice's 8
//             MMAs, so a slot's MMAs are issued in half the time and the SM issues twice as many
//   V_WIDE:   batched-layout normal tiles of 256 token rows (two 128-row MMA halves sharing each B stage):
//             smem [A rows 0..127 16 KB][A rows 128..255 16 KB][B 32 KB] x 3 stages; TMEM: one accumulator of
//             two 256-column halves (the whole 512 columns, so no second buffer); 320 threads (8 epilogue
//             warps, one per TMEM lane quarter and half).  Each stage carries twice the MMA work of a V_BF16
//             stage for 4/3 of its bytes.
enum { V_BF16 = 0, V_E4M3 = 1, V_SWAP64 = 2, V_WIDE = 3, V_E4M3N = 4 };

template <int V>
struct Cfg {
    static constexpr bool W8 = V == V_E4M3 || V == V_E4M3N;
    static constexpr bool E4N = V == V_E4M3N;
    static constexpr bool NARROW = V == V_SWAP64;
    static constexpr bool WIDE = V == V_WIDE;
    static constexpr int KSUB = W8 ? 2 : 1;                     // 64-wide k-blocks per stage
    static constexpr int STAGES = W8 ? (E4N ? 11 : 9) : (NARROW ? 8 : (WIDE ? 3 : 4));   // E4M3: code stages
    static constexpr int A_PARTS = WIDE ? 2 : 1;                // 128-row A tiles per stage
    static constexpr int A_SLOTS = 4;                           // E4M3: TMEM A tiles (+ token tiles)
    static constexpr int TOK_SPAN = E4N ? 32 : ((W8 || NARROW) ? 64 : 256);   // swap-AB tokens per tile
    static constexpr int B_OFF = W8 ? 0 : A_PARTS * A_BYTES;    // bf16: B operand offset in a stage
    static constexpr int B_SUB = TOK_SPAN * BK * 2;             // token bytes per 64-wide k-block (swap)
    static constexpr int B_BYTES = W8 ? 0 : (NARROW ? B_SUB : 256 * BK * 2);
    static constexpr int STAGE_BYTES = W8 ? BM * BK * KSUB : A_PARTS * A_BYTES + B_BYTES;
    static constexpr int TOK_OFF = STAGES * STAGE_BYTES;        // E4M3: token slots after the code ring
    static constexpr int TOK_SLOT = B_SUB * KSUB;
    static constexpr int EPI_WARPS = WIDE ? 8 : 4;
    static constexpr int ISSUERS = E4N ? 4 : (W8 ? 2 : 1);     // MMA-issuing warps, one accumulator each
    static constexpr int PER_SLICE = W8 ? ISSUERS / 2 : 1;      // E4M3: issuers sharing a slice's MMAs
    static constexpr int THREADS = W8 ? 192 + kConvThreads + 32 * (ISSUERS - 1) : 64 + 32 * EPI_WARPS;
    static constexpr int MMA2_WARP = 6 + kConvThreads / 32;     // E4M3: first MMA warp after warp 1
    static constexpr int SMEM = STAGES * STAGE_BYTES + (W8 ? A_SLOTS * TOK_SLOT : 0) + 1024;
    static constexpr int ACC_STRIDE = (W8 || NARROW) ? TOK_SPAN : ACC_COLS; // TMEM columns per accumulator (half)
    static constexpr int NBUF = WIDE ? 1 : 2;                   // accumulators (the wide one fills TMEM)
    static constexpr int A_TMEM = 2 * ISSUERS * ACC_STRIDE;     // E4M3: first A tile column
    static constexpr int A_COLS = KSUB * BK / 2;                // E4M3: TMEM columns per A tile
    static constexpr int TMEM_USED = W8 ? A_TMEM + A_SLOTS * A_COLS : (WIDE ? 2 * ACC_COLS : 2 * ACC_STRIDE);
};
static_assert(Cfg<V_BF16>::TMEM_USED <= TMEM_COLS, "bf16 accumulators exceed the TMEM allocation");
static_assert(Cfg<V_SWAP64>::TMEM_USED <= TMEM_COLS, "bf16 accumulators exceed the TMEM allocation");
static_assert(Cfg<V_WIDE>::TMEM_USED <= TMEM_COLS, "bf16 accumulators exceed the TMEM allocation");
static_assert(Cfg<V_WIDE>::SMEM + 13 * 1024 <= 227 * 1024, "bf16 stage ring exceeds shared memory");
static_assert(Cfg<V_E4M3>::TMEM_USED <= TMEM_COLS, "E4M3 accumulators and A tiles exceed the TMEM allocation");
static_assert(Cfg<V_E4M3N>::TMEM_USED <= TMEM_COLS, "E4M3 accumulators and A tiles exceed the TMEM allocation");
static_assert(Cfg<V_E4M3N>::SMEM + 13 * 1024 <= 227 * 1024, "E4M3 stage ring exceeds shared memory");
static_assert(Cfg<V_E4M3N>::STAGES <= MAX_STAGES, "too many stages");
static_assert(Cfg<V_BF16>::SMEM + 13 * 1024 <= 227 * 1024, "bf16 stage ring exceeds shared memory");
static_assert(Cfg<V_SWAP64>::SMEM + 13 * 1024 <= 227 * 1024, "bf16 stage ring exceeds shared memory");
static_assert(Cfg<V_E4M3>::SMEM + 13 * 1024 <= 227 * 1024, "E4M3 stage ring exceeds shared memory");
static_assert(Cfg<V_E4M3>::STAGES <= MAX_STAGES && Cfg<V_BF16>::STAGES <= MAX_STAGES &&
                  Cfg<V_SWAP64>::STAGES <= MAX_STAGES,
              "too many stages");
static_assert(Cfg<V_E4M3>::A_SLOTS == 4, "converter groups take A slot (stage index mod 4)");

struct __align__(8) Ctrl {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t conv[MAX_STAGES];   // E4M3: A slot converted and its tokens copied
    uint64_t a_empty[4];         // E4M3: A slot free (MMA done)
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    volatile int abort;
};

struct TcParams {
    int gemm;            // 1 or 2
    int swap;            // 0 normal, 1 swap-AB
    int layout;
    int E;
    int max_tokens;
    int64_t rows_cap;
    int nkb;             // k-blocks per tile
    int nt;              // normal: n-tiles per m-tile; swap: weight blocks per expert
    int w_mode;          // weights map: 0 = 3-D (k, rows, E), 1 = 5-D gate/up interleaving view,
                         // 2 = 4-D tile-contiguous (64, 128, k-blocks, E x 128-row blocks; swap-AB tiles)
    int64_t I, K;
    const int32_t* counts;
    const int32_t* offsets;
    const int32_t* row_route;
    const float* route_w;
    void* out;
    int out_dtype;
    int64_t out_rows;    // GEMM 2, contiguous: rows of y (routes)
    int32_t* err_word;
    int span;            // activation rows per tile (normal: 128; swap: token segment)
    int mixed;           // 1: normal tiles plus a swap-AB tile for each expert's short tail
    int nt_n, nt_s;      // mixed: weight tiles per m-tile (normal, 256 rows) and per segment (swap, 128 rows)
    const uint8_t* w_scale;   // E4M3 weights: E8M0 scales (E, wrows, kdim/32)
    const uint16_t* act;      // E4M3 weights: bf16 activation rows (rows_cap, act_ld), copied by the converters
    int64_t act_ld;
    int64_t wrows;       // weight rows per expert
    int64_t nsb;         // scale bytes per weight row (kdim / 32)
    int skip_first_copy; // test hook: CTA 0 never issues its first weight copy (see timeout_test_hook)
    // fused experts (GEMM 1 tiles, then GEMM 2 tiles, in one launch; bf16 swap-AB tiles, contiguous layout):
    // tm_act/tm_w map x rows and W1, tm_act_s/tm_w_s map h and W2; out is h, out2 is y
    int fused;
    int nkb2, nt2;       // GEMM 2: k-blocks per tile, weight blocks per expert
    int w_mode2;         // GEMM 2: weights map (0 or 2)
    void* out2;
    int out2_dtype;
    int32_t* seg_done;   // per token segment: GEMM 1 epilogue warps done (zero at launch)
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

// Fused launches: waits until *ctr >= need (GEMM 1 epilogue warps of a token segment have published h), read
// with acquire semantics at GPU scope; bounded like every other wait.
MOE_DEVICE bool wait_counter(const int32_t* ctr, int32_t need, Ctrl& c, int32_t* err_word) {
    const uint64_t deadline = ptx::globaltimer() + kWaitNs;
    uint32_t n = 0;
    while (true) {
        int32_t v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= need) return true;
        if ((++n & 255u) == 0) {
            if (c.abort) return false;
            if (ptx::globaltimer() > deadline) {
                c.abort = 1;
                report(err_word, MOE_DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Tile -> (expert, rows, n-tile / weight block, tokens) decoding, shared by all roles.
struct Tile {
    int gemm;         // 1 or 2 (fused launches hold both)
    int32_t seg;      // fused: global token-segment index
    int swap;         // this tile puts weights on the MMA M side
    int e;
    int64_t row0;     // first activation row of the tile
    int rows;         // valid activation rows (normal: <= 128; swap: tokens <= 256)
    int nb;           // normal: n-tile; swap: weight block
};

// Mixed mode: an expert with at least 64 rows gets normal 128-row m-tiles (the last one padded); a smaller
// expert gets one swap-AB segment instead.  Either way each expert's weights are streamed once: a swap-AB
// tile for the tail of a large expert would stream them a second time, which costs more than the padding.
MOE_DEVICE int mixed_normal_tiles(int32_t c) { return c >= 64 ? (c + BM - 1) / BM : 0; }
MOE_DEVICE int32_t mixed_tail(int32_t c) { return c >= 64 ? 0 : c; }

MOE_DEVICE Tile decode_tile(const ExpertTable& tab, const TcParams& p, int32_t t) {
    Tile tl;
    tl.gemm = p.gemm;
    tl.seg = 0;
    if (p.fused) {
        // the table counts token segments; GEMM 1 tiles (segment, W1 block) come first, then GEMM 2 tiles
        const int32_t t1 = tab.total * p.nt;
        int32_t tt = t, nt = p.nt;
        if (t >= t1) {
            tl.gemm = 2;
            tt = t - t1;
            nt = p.nt2;
        } else {
            tl.gemm = 1;
        }
        const int32_t g = tt / nt;
        tl.seg = g;
        tl.nb = tt - g * nt;
        tl.e = find_expert(tab, p.E, g);
        const int32_t seg = g - tiles_before(tab, tl.e);
        tl.swap = 1;
        tl.row0 = int64_t(tab.start[tl.e]) + int64_t(seg) * p.span;
        tl.rows = min(p.span, tab.count[tl.e] - seg * p.span);
        return tl;
    }
    tl.e = find_expert(tab, p.E, t);
    const int32_t local = t - tiles_before(tab, tl.e);
    if (p.mixed) {
        const int32_t c = tab.count[tl.e];
        const int32_t nn = mixed_normal_tiles(c);
        if (local < nn * p.nt_n) {
            const int32_t m = local / p.nt_n;
            tl.swap = 0;
            tl.nb = local - m * p.nt_n;
            tl.row0 = int64_t(tab.start[tl.e]) + int64_t(m) * BM;
            tl.rows = min(BM, c - m * BM);
        } else {
            tl.swap = 1;
            tl.nb = local - nn * p.nt_n;
            tl.row0 = int64_t(tab.start[tl.e]);
            tl.rows = mixed_tail(c);
        }
        return tl;
    }
    tl.swap = p.swap;
    const int32_t seg = local / p.nt;
    tl.nb = local - seg * p.nt;
    tl.row0 = int64_t(tab.start[tl.e]) + int64_t(seg) * p.span;
    tl.rows = min(p.span, tab.count[tl.e] - seg * p.span);
    return tl;
}

// The k-th tile of CTA b among G CTAs.  Fused launches walk the tiles serpentine (b, 2G-1-b, 2G+b, ...): their
// list holds all GEMM 1 tiles (K-long weight rows) before the GEMM 2 tiles (I-long rows), so plain round-robin
// hands the CTAs of low index more bytes; measured on the decode sweep, the serpentine order is 0.6 % faster
// (1.5 % at T=8), while on the MXFP8-weight tiles, all of one size, it was 1.4 % slower.
MOE_DEVICE int32_t nth_tile(const TcParams& p, int32_t k) {
    const int32_t G = int32_t(gridDim.x), b = int32_t(blockIdx.x);
    return k * G + ((p.fused && (k & 1)) ? G - 1 - b : b);
}

// Weight row (within the expert) held by row r of a 128-row swap-AB weight tile nb.
MOE_DEVICE int64_t tile_weight_row(const TcParams& p, int nb, int r) {
    if (p.w_mode == 1) {   // [gate; up] rows seen through the interleave-16 view
        const int64_t unit = int64_t(nb) * 64 + (r >> 5) * 16 + (r & 15);
        return ((r >> 4) & 1) * p.I + unit;
    }
    return int64_t(nb) * 128 + r;
}

// Normal-tile GEMM 1 epilogue, one 32-column chunk c of a row: columns [gate16, up16] of units
// 128*nb + 16*c .. +15 -> 16 bf16 values of h.
MOE_DEVICE void store_h_chunk(const TcParams& p, const uint32_t (&v)[32], bool valid, int64_t row, int nb, int c) {
    if (!valid) return;
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float h0 = silu_mul(__uint_as_float(v[2 * i]), __uint_as_float(v[16 + 2 * i]));
        const float h1 = silu_mul(__uint_as_float(v[2 * i + 1]), __uint_as_float(v[16 + 2 * i + 1]));
        o[i] = pack_bf16x2(h0, h1);
    }
    const int64_t unit = int64_t(nb) * 128 + c * 16;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row * p.I + unit);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// Normal-tile GEMM 2 epilogue, one 32-column chunk c of a row: weight times the 32 outputs, written to the
// route's row of y.
MOE_DEVICE void store_y_chunk(const TcParams& p, const uint32_t (&v)[32], int64_t dst_row, float wt, int nb, int c) {
    if (dst_row < 0) return;
    const int64_t col = int64_t(nb) * 256 + c * 32;
    if (p.out_dtype == MOE_BF16) {
        uint32_t o[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = pack_bf16x2(wt * __uint_as_float(v[2 * i]), wt * __uint_as_float(v[2 * i + 1]));
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + dst_row * p.K + col);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    } else {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + dst_row * p.K + col);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(wt * __uint_as_float(v[4 * i]), wt * __uint_as_float(v[4 * i + 1]),
                                 wt * __uint_as_float(v[4 * i + 2]), wt * __uint_as_float(v[4 * i + 3]));
    }
}

// E4M3 converter, one weight row of a slice: its 128 codes (at `row`, landed 128-byte swizzled: 16-byte chunk c
// of row r at chunk c ^ (r % 8)) times the four block scales in `quad` (block b in byte b) -> 64 bf16x2 words
// in TMEM columns tmem .. tmem + 63 of this thread's lane.  BIG: a scale code of the warp is above 134, so a
// block may need the second multiply by 2^120; otherwise the four factors come from the scale word at once.
template <bool BIG>
MOE_DEVICE void decode_row_slice(const uint8_t* row, int r, uint32_t quad, uint32_t tmem) {
    const uint32_t q120 = quad + 0x78787878u;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        uint32_t o[32];
#pragma unroll
        for (int b2 = 0; b2 < 2; ++b2) {
            const int b = 2 * half + b2;     // scale block of the slice
            bool second = false;             // the factor 2^120 still to apply (large scales)
            const uint32_t f1 = BIG ? mx_e4m3_factor((quad >> (8 * b)) & 0xFFu, second) : mx_e4m3_factor_small(q120, b);
            const uint4 v0 = *reinterpret_cast<const uint4*>(row + (((2 * b) ^ (r & 7)) << 4));
            const uint4 v1 = *reinterpret_cast<const uint4*>(row + (((2 * b + 1) ^ (r & 7)) << 4));
            uint32_t* ob = o + 16 * b2;
            dequant4(v0.x, f1, ob[0], ob[1]);
            dequant4(v0.y, f1, ob[2], ob[3]);
            dequant4(v0.z, f1, ob[4], ob[5]);
            dequant4(v0.w, f1, ob[6], ob[7]);
            dequant4(v1.x, f1, ob[8], ob[9]);
            dequant4(v1.y, f1, ob[10], ob[11]);
            dequant4(v1.z, f1, ob[12], ob[13]);
            dequant4(v1.w, f1, ob[14], ob[15]);
            if (BIG && second) {
#pragma unroll
                for (int i = 0; i < 16; ++i) ob[i] = bf16x2_mul(ob[i], kBf16x2Pow2_120);
            }
        }
        ptx::tmem_st_32x32b_x32(tmem + uint32_t(half * 32), o);
    }
}

template <int V>
__global__ void __launch_bounds__(Cfg<V>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_w,
                   const __grid_constant__ CUtensorMap tm_act_s, const __grid_constant__ CUtensorMap tm_w_s,
                   const TcParams p) {
    // tm_act/tm_w: boxes of normal tiles (or of every tile when all tiles are of one kind);
    // tm_act_s/tm_w_s: boxes of the swap-AB tiles of a mixed launch
    constexpr bool W8 = Cfg<V>::W8;
    constexpr int STAGES = Cfg<V>::STAGES;
    constexpr int STAGE_BYTES = Cfg<V>::STAGE_BYTES;
    if constexpr (Cfg<V>::NARROW) {
        if (!p.swap || p.mixed) return;   // the narrow ring holds swap-AB tiles only (the host never asks more)
    }
    if constexpr (Cfg<V>::WIDE) {
        if (p.swap || p.mixed || p.fused) return;   // normal tiles only (the host never asks more)
    }
    extern __shared__ uint8_t smem_raw[];
    __shared__ ExpertTable tab;
    __shared__ Ctrl ctrl;
    // E4M3: the producer hands each tile it decodes to the converter warps through a 4-entry ring, so that the
    // tile look-up is off the converters' path (measured: 0.8 us per tile there, 10 % of a 16-slice tile)
    __shared__ Tile tinfo[4];
    __shared__ uint64_t tinfo_full[4], tinfo_empty[4];

    // 1024-byte aligned stage buffers (the 128-byte swizzle pattern repeats every 1024 bytes)
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&ctrl.full[s], 1);
            ptx::mbar_init(&ctrl.empty[s], W8 ? 4 : 1);   // E4M3: freed by the 4 warps of the converting group
        }
        for (int a = 0; a < Cfg<V>::A_SLOTS; ++a) {
            ptx::mbar_init(&ctrl.conv[a], 4);             // the 4 converter warps of the slot's group
            ptx::mbar_init(&ctrl.a_empty[a], Cfg<V>::PER_SLICE);   // E4M3: each issuer of the slice commits
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&ctrl.acc_full[b], Cfg<V>::ISSUERS);   // one commit per MMA issuer
            ptx::mbar_init(&ctrl.acc_empty[b], Cfg<V>::EPI_WARPS);
        }
        ptx::mbar_init(&ctrl.drain, Cfg<V>::ISSUERS);
        for (int i = 0; i < 4; ++i) {
            ptx::mbar_init(&tinfo_full[i], 1);                    // the producer wrote the entry
            ptx::mbar_init(&tinfo_empty[i], kConvThreads / 32);   // every converter warp read it
        }
        ctrl.abort = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tm_act);
        ptx::prefetch_tmap(&tm_w);
        if (p.mixed) {
            ptx::prefetch_tmap(&tm_act_s);
            ptx::prefetch_tmap(&tm_w_s);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc(&ctrl.tmem_base, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    const int span = p.span, ntl = p.fused ? 1 : p.nt, mixed = p.mixed, ntn = p.nt_n, nts = p.nt_s;
    build_expert_table(tab, p.E, p.counts, p.offsets, p.max_tokens, p.rows_cap,
                       [span, ntl, mixed, ntn, nts](int32_t c) {
                           if (mixed) return mixed_normal_tiles(c) * ntn + (mixed_tail(c) > 0 ? nts : 0);
                           return ((c + span - 1) / span) * ntl;
                       });
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = ctrl.tmem_base;
    const int32_t total = p.fused ? tab.total * (p.nt + p.nt2) : tab.total;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // L2 hints: swap-AB weights are streamed once (evict first); normal-tile weights are reused by
            // every m-tile of the expert and activation rows by every n-tile (keep them)
            const uint64_t pol_stream = ptx::policy_evict_first();
            const uint64_t pol_keep = ptx::policy_evict_last();
            const uint64_t pol_a = pol_keep;
            uint32_t it = 0;
            for (int32_t k_ = 0, t = blockIdx.x; t < total && !ctrl.abort; t = nth_tile(p, ++k_)) {
                const Tile tl = decode_tile(tab, p, t);
                if constexpr (W8) {   // the tile for the converters (entry k % 4, reused once all 16 warps read it)
                    const int ts = k_ & 3;
                    if (!wait_bar(&tinfo_empty[ts], ((k_ >> 2) & 1) ^ 1, ctrl, p.err_word)) break;
                    tinfo[ts] = tl;
                    ptx::mbar_arrive(&tinfo_full[ts]);
                }
                const int nbox = tl.swap ? (tl.rows + TOK_BOX - 1) / TOK_BOX : 0;
                const bool second = (p.mixed && tl.swap) || (tl.gemm == 2 && p.fused);   // maps of the second kind
                const CUtensorMap* mact = second ? &tm_act_s : &tm_act;
                const CUtensorMap* mw = second ? &tm_w_s : &tm_w;
                const int nkb = tl.gemm == 2 && p.fused ? p.nkb2 : p.nkb;
                const int w_mode = tl.gemm == 2 && p.fused ? p.w_mode2 : p.w_mode;
                const int wblocks = tl.gemm == 2 && p.fused ? p.nt2 : p.nt;   // 128-row weight blocks per expert
                if (p.fused && tl.gemm == 2) {
                    // this segment's h is complete once all 4 epilogue warps of its nt GEMM 1 tiles published
                    if (!wait_counter(&p.seg_done[tl.seg], 4 * p.nt, ctrl, p.err_word)) break;
                    asm volatile("fence.proxy.async.global;" ::: "memory");   // generic writes -> TMA reads
                }
                const uint64_t pol_w = tl.swap ? pol_stream : pol_keep;
                constexpr int KSUB = Cfg<V>::KSUB;
                const uint32_t wbytes = W8 ? uint32_t(BM * BK * KSUB) : uint32_t(A_BYTES);
                const int aparts = (Cfg<V>::WIDE && tl.rows > BM) ? 2 : 1;   // wide tiles: second row half used
                const uint32_t bytes = W8 ? wbytes
                                          : (tl.swap ? wbytes + uint32_t(nbox * TOK_BOX * BK * 2)
                                                     : uint32_t(aparts * A_BYTES + Cfg<V>::B_BYTES));
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!wait_bar(&ctrl.empty[s], ph ^ 1, ctrl, p.err_word)) break;
                    uint8_t* sa = smem + s * STAGE_BYTES;
                    uint8_t* sb = sa + Cfg<V>::B_OFF;
                    ptx::mbar_arrive_expect_tx(&ctrl.full[s], bytes);
                    if (p.skip_first_copy && blockIdx.x == 0 && it == 0) continue;   // bytes that never arrive
                    const int k0 = kb * BK * KSUB;
                    // weights: normal -> B operand (256 rows); swap -> A operand (128 rows);
                    // E4M3 codes -> 128-byte rows for the converters
                    uint8_t* wdst = W8 ? sa : (tl.swap ? sa : sb);
                    const int wrows = tl.swap ? 128 : 256;
                    const int row_w = tl.nb * wrows;          // first weight row (interleaved order)
                    if (w_mode == 1)
                        ptx::tma_load_5d(wdst, mw, &ctrl.full[s], k0, 0, 0, row_w / 32, tl.e, pol_w);
                    else if (w_mode == 2)   // one contiguous 16 KB block per k-block
                        ptx::tma_load_4d(wdst, mw, &ctrl.full[s], 0, 0, kb, tl.e * wblocks + tl.nb, pol_w);
                    else
                        ptx::tma_load_3d(wdst, mw, &ctrl.full[s], k0, row_w, tl.e, pol_w);
                    if (W8) {
                        // E4M3: the converters copy the tokens
                    } else if (tl.swap) {
                        for (int b = 0; b < nbox; ++b)
                            ptx::tma_load_2d(sb + b * TOK_BOX * BK * 2, mact, &ctrl.full[s], k0,
                                             int32_t(tl.row0 + b * TOK_BOX), pol_a);
                    } else {
                        ptx::tma_load_2d(sa, mact, &ctrl.full[s], k0, int32_t(tl.row0), pol_a);
                        if (aparts == 2)
                            ptx::tma_load_2d(sa + A_BYTES, mact, &ctrl.full[s], k0, int32_t(tl.row0 + BM), pol_a);
                    }
                }
            }
            // let every copy issued so far land before the CTA can exit
            const uint32_t issued = it;
            for (uint32_t j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j) {
                const int s = j % STAGES;
                const uint64_t deadline = ptx::globaltimer() + kWaitNs / 4;
                volatile int never = 0;
                ptx::mbar_wait_bounded(&ctrl.full[s], (j / STAGES) & 1, deadline, &never);
            }
        }
        __syncwarp();
    } else if (warp == 1 || (W8 && warp >= Cfg<V>::MMA2_WARP && warp < Cfg<V>::MMA2_WARP + Cfg<V>::ISSUERS - 1)) {
        // ------------------------------------------------------------ MMA issuer
        // E4M3: issuer j (warp 1: j = 0, the further MMA warps: j = 1, 2, ...) takes the k slices of parity
        // j / PER_SLICE of every tile, and of each such slice the MMAs of part j % PER_SLICE, into accumulator j
        // of the buffer; bf16 variants have one issuer.  The whole warp runs the loop (waits, addresses and
        // descriptors are warp-uniform) and lane 0 issues every MMA and commit.
        const int j = warp == 1 ? 0 : warp - Cfg<V>::MMA2_WARP + 1;
        const int par = j / Cfg<V>::PER_SLICE, part = j % Cfg<V>::PER_SLICE;
        const uint32_t issue = lane == 0;
        uint32_t it = 0, tc = 0;
        for (int32_t k_ = 0, t = blockIdx.x; t < total && !ctrl.abort; t = nth_tile(p, ++k_), ++tc) {
            const Tile tl = decode_tile(tab, p, t);
            const int buf = Cfg<V>::NBUF == 2 ? int(tc & 1) : 0;
            const uint32_t aph = Cfg<V>::NBUF == 2 ? (tc >> 1) & 1 : tc & 1;
            if (!__all_sync(0xffffffffu, wait_bar(&ctrl.acc_empty[buf], aph ^ 1, ctrl, p.err_word))) break;
            ptx::tc_fence_after();
            const bool half2 = Cfg<V>::WIDE && tl.rows > BM;   // wide tiles: MMAs for rows 128..255
            int n_mma = 256;
            if (tl.swap) n_mma = max(16, (tl.rows + 15) / 16 * 16);
            const uint32_t idesc = ptx::idesc_bf16(BM, n_mma);
            const uint32_t d_tmem = tmem_base + uint32_t((buf * Cfg<V>::ISSUERS + j) * Cfg<V>::ACC_STRIDE);
            const int nkb = tl.gemm == 2 && p.fused ? p.nkb2 : p.nkb;
            bool ok = true;
            if constexpr (W8) {
                // this issuer's slices of the tile: kb = par, par + 2, ...; A slot and parity of slice it0 + kb
                const uint32_t it0 = it;
                for (int kb = par; kb < nkb; kb += 2) {
                    const uint32_t itk = it0 + uint32_t(kb);
                    const int a = int(itk & 3u);
                    const uint32_t ph = (itk >> 2) & 1u;
                    if (!__all_sync(0xffffffffu, wait_bar(&ctrl.conv[a], ph, ctrl, p.err_word))) { ok = false; break; }
                    ptx::tc_fence_after();
                    // tokens in the slot's smem tile (descriptor start addresses step by 16 bytes), decoded weights in
                    // the slot's TMEM columns
                    const uint64_t bd0 = ptx::smem_desc_sw128(ptx::smem_addr(smem + Cfg<V>::TOK_OFF + a * Cfg<V>::TOK_SLOT));
                    const uint32_t a0 = tmem_base + uint32_t(Cfg<V>::A_TMEM + a * Cfg<V>::A_COLS);
                    constexpr int KK = Cfg<V>::KSUB * BK / UMMA_K / Cfg<V>::PER_SLICE;   // MMAs per issuer
#pragma unroll
                    for (int k2 = 0; k2 < KK; ++k2) {
                        const int kk = part * KK + k2;   // k step of the slice
                        const int sub = kk / (BK / UMMA_K), kq = kk % (BK / UMMA_K);
                        const uint64_t bd = bd0 + uint64_t((sub * Cfg<V>::B_SUB + kq * UMMA_K * 2) >> 4);
                        // 16 bf16 of a row = 8 TMEM columns per k step
                        ptx::mma_f16_tmem_a_by(issue, d_tmem, a0 + uint32_t(kk * 8), bd, idesc, kb != par || k2 != 0);
                    }
                    ptx::mma_commit_by(issue, &ctrl.a_empty[a]);
                }
                it += uint32_t(nkb);
            } else {
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!__all_sync(0xffffffffu, wait_bar(&ctrl.full[s], ph, ctrl, p.err_word))) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_addr(smem + s * STAGE_BYTES);
                    const uint32_t sb = sa + Cfg<V>::B_OFF;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        const uint64_t ad = ptx::smem_desc_sw128(sa + kk * UMMA_K * 2);
                        const uint64_t bd = ptx::smem_desc_sw128(sb + kk * UMMA_K * 2);
                        ptx::mma_f16_by(issue, d_tmem, ad, bd, idesc, (kb | kk) != 0);
                        if (half2) {
                            const uint64_t ad2 = ptx::smem_desc_sw128(sa + A_BYTES + kk * UMMA_K * 2);
                            ptx::mma_f16_by(issue, d_tmem + ACC_COLS, ad2, bd, idesc, (kb | kk) != 0);
                        }
                    }
                    ptx::mma_commit_by(issue, &ctrl.empty[s]);
                }
            }
            if (!ok) break;
            ptx::mma_commit_by(issue, &ctrl.acc_full[buf]);
        }
        // all MMAs issued by lane 0 complete before TMEM is released
        ptx::mma_commit_by(issue, &ctrl.drain);
        const uint64_t deadline = ptx::globaltimer() + kWaitNs / 4;
        volatile int never = 0;
        ptx::mbar_wait_bounded(&ctrl.drain, 0, deadline, &never);
        __syncwarp();
    } else if (W8 && warp >= 6) {
        // ------------------------------------------------------------ E4M3 converters
        // Four groups of 4 warps take stages in turn (group = stage index mod 4 = its A slot), so four
        // stages are in conversion at once.  In a group, thread (warp w, lane) owns row r = 32*(w%4) + lane
        // of the 128-row weight tile: its 128 codes of the slice (scale blocks 0..3) go to TMEM lane r, the
        // slot's 64 A-tile columns.  The group also copies the slice's token rows into the slot.
        const int cw = warp - 6, grp = cw >> 2;
        const int q = warp & 3, r = q * 32 + lane;
        const uint32_t lane_base = uint32_t(q * 32) << 16;
        const bool vec_scales = (p.nsb & 15) == 0;       // 16-byte aligned scale rows (4 slices per 16 B)
        const uint64_t pol_keep = ptx::policy_evict_last();   // token rows are read by every weight block
        uint32_t it = 0;
        // this group's slices are it = grp, grp + 4, ...: their code stage (it % STAGES) and the parities of the
        // code ring and of the A slot advance incrementally
        int s_own = grp;
        uint32_t ph_own = 0, pha_own = 0, it_next = uint32_t(grp);
        for (int32_t k_ = 0, t = blockIdx.x; t < total && !ctrl.abort; t = nth_tile(p, ++k_)) {
            const int ts = k_ & 3;   // the tile as the producer decoded it
            if (!wait_bar(&tinfo_full[ts], (k_ >> 2) & 1, ctrl, p.err_word)) break;
            const Tile tl = tinfo[ts];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&tinfo_empty[ts]);
            const uint8_t* srow = p.w_scale + (int64_t(tl.e) * p.wrows + tile_weight_row(p, tl.nb, r)) * p.nsb;
            // this thread's 16-byte token chunks of a slice: column chunk r % 8 of k-block half (r / 8) % 2, rows
            // n = r / 16 + 8j of the tile (the slot's chunks in order, 128 threads apart), so only the row and
            // the slice's k offset change from chunk to chunk
            const int n0 = r >> 4, tsub = (r >> 3) & 1, tcc = r & 7;
            const int nrow16 = (tl.rows + TOK_BOX - 1) / TOK_BOX * TOK_BOX;   // rows past tl.rows are zero-filled
            const uint16_t* tok0 = p.act + tl.row0 * p.act_ld + tsub * BK + tcc * 8;   // tile row 0
            const uint32_t tok_dst = uint32_t(tsub * Cfg<V>::B_SUB + n0 * (BK * 2) + ((tcc ^ (n0 & 7)) << 4));
            bool ok = true;
            for (int kb = int(it_next - it); kb < p.nkb; kb += 4) {
                uint32_t quad;                      // this row's four scale bytes of the slice
                if (vec_scales) {
                    quad = __ldg(reinterpret_cast<const uint32_t*>(srow + 4 * kb));
                } else {
                    quad = 0;
                    for (int b = 0; b < 4; ++b) quad |= uint32_t(__ldg(srow + 4 * kb + b)) << (8 * b);
                }
                if (kb + 16 < p.nkb) asm volatile("prefetch.global.L1 [%0];" ::"l"(srow + 4 * (kb + 16)));
                const int s = s_own, a = grp;
                const uint32_t ph = ph_own, pha = pha_own;
                s_own += 4;
                if (s_own >= STAGES) {
                    s_own -= STAGES;
                    ph_own ^= 1;
                }
                pha_own ^= 1;
                it_next += 4;
                if (!wait_bar(&ctrl.a_empty[a], pha ^ 1, ctrl, p.err_word)) { ok = false; break; }
                ptx::tc_fence_after();   // the MMA that last read this A slot has completed
                {
                    // the slice's token rows -> the slot's two 64-wide k-blocks, rows of 128 bytes, 16-byte chunk
                    // c of row n at chunk c ^ (n % 8) (the 128-byte swizzle of the MMA's B operand; n % 8 is the
                    // same for all of this thread's rows); rows past the tile's tokens are zero-filled without a
                    // global read
                    const uint32_t dst = ptx::smem_addr(smem + Cfg<V>::TOK_OFF + a * Cfg<V>::TOK_SLOT) + tok_dst;
                    const uint16_t* src0 = tok0 + int64_t(kb) * BK * Cfg<V>::KSUB;
#pragma unroll
                    for (int j = 0; j < Cfg<V>::TOK_SPAN / 8; ++j) {
                        const int n = n0 + 8 * j;
                        if (n < nrow16) {
                            const bool valid = n < tl.rows;
                            ptx::cp_async_16(dst + uint32_t(j * 8 * BK * 2), valid ? src0 + int64_t(n) * p.act_ld : src0,
                                             valid ? 16u : 0u, pol_keep);
                        }
                    }
                }
                if (!wait_bar(&ctrl.full[s], ph, ctrl, p.err_word)) {
                    ptx::cp_async_wait_all();   // no copy of this thread is left in flight
                    ok = false;
                    break;
                }
                const uint8_t* row = smem + s * STAGE_BYTES + r * (BK * 2);
                const uint32_t a_cols = tmem_base + lane_base + uint32_t(Cfg<V>::A_TMEM + a * Cfg<V>::A_COLS);
                if (__any_sync(0xffffffffu, mx_scale_above_134(quad) != 0))
                    decode_row_slice<true>(row, r, quad, a_cols);
                else
                    decode_row_slice<false>(row, r, quad, a_cols);
                ptx::tmem_st_wait();
                ptx::cp_async_wait_all();           // this thread's token copies have landed
                ptx::fence_proxy_async_smem();      // and are visible to the MMA's operand reads
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    ptx::mbar_arrive(&ctrl.empty[s]);   // the code stage can be refilled
                    ptx::mbar_arrive(&ctrl.conv[a]);    // the A slot and its tokens are ready for the MMA
                }
            }
            it += uint32_t(p.nkb);
            if (!ok) break;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                       // TMEM lane quarter of this warp
        const int half = Cfg<V>::WIDE ? (warp - 2) >> 2 : 0;   // wide tiles: row half of this warp
        const uint32_t lane_base = uint32_t(q * 32) << 16;
        uint32_t tc = 0;
        for (int32_t k_ = 0, t = blockIdx.x; t < total; t = nth_tile(p, ++k_), ++tc) {
            const Tile tl = decode_tile(tab, p, t);
            const int buf = Cfg<V>::NBUF == 2 ? int(tc & 1) : 0;
            const uint32_t aph = Cfg<V>::NBUF == 2 ? (tc >> 1) & 1 : tc & 1;
            if (!wait_bar(&ctrl.acc_full[buf], aph, ctrl, p.err_word)) break;
            ptx::tc_fence_after();
            const uint32_t tacc =
                tmem_base + lane_base + uint32_t(buf * Cfg<V>::ISSUERS * Cfg<V>::ACC_STRIDE + half * ACC_COLS);
            if (!tl.swap) {
              if constexpr (V == V_BF16 || V == V_WIDE) {   // the other variants run swap-AB tiles only
               if (half * BM < tl.rows) {                     // (a wide tile may have no second half)
                const int r = half * BM + q * 32 + lane;      // tile row of this thread
                const bool valid = r < tl.rows;
                const int64_t row = tl.row0 + r;
                int64_t dst_row = -1;                         // GEMM 2: destination row, weight
                float wt = 1.f;
                if (p.gemm == 2 && valid) {
                    if (p.layout == MOE_LAYOUT_CONTIGUOUS) {
                        const int32_t route = p.row_route[row];
                        if (route >= 0 && route < p.out_rows) {
                            dst_row = route;
                            if (p.route_w) wt = p.route_w[route];
                        }
                    } else {
                        dst_row = row;
                        if (p.route_w) wt = p.route_w[row];
                    }
                }
                // 8 chunks of 32 columns; chunk c + 1 is read from TMEM while chunk c is converted and stored
                uint32_t va[32], vb[32];
                ptx::tmem_ld_32x32b_x32(tacc, va);
                ptx::tmem_ld_wait_regs(va);
#pragma unroll 1
                for (int c = 0; c < ACC_COLS / 32; c += 2) {
                    ptx::tmem_ld_32x32b_x32(tacc + (c + 1) * 32, vb);
                    if (p.gemm == 1) store_h_chunk(p, va, valid, row, tl.nb, c);
                    else store_y_chunk(p, va, dst_row, wt, tl.nb, c);
                    ptx::tmem_ld_wait_regs(vb);
                    if (c + 2 < ACC_COLS / 32) ptx::tmem_ld_32x32b_x32(tacc + (c + 2) * 32, va);
                    if (p.gemm == 1) store_h_chunk(p, vb, valid, row, tl.nb, c + 1);
                    else store_y_chunk(p, vb, dst_row, wt, tl.nb, c + 1);
                    if (c + 2 < ACC_COLS / 32) ptx::tmem_ld_wait_regs(va);
                }
               }
              }
            } else {
                // swap-AB: TMEM lane = weight row of the tile, column = token
                const int n_tok = tl.rows;
                const int n_chunks = (n_tok + 15) / 16;
                // 16 token columns of this thread's row; E4M3: the accumulators of all issuers added (those of
                // the odd-slice issuers hold something when the tile has two or more slices)
                const int n_acc = (Cfg<V>::ISSUERS > 1 && p.nkb < 2) ? Cfg<V>::PER_SLICE : Cfg<V>::ISSUERS;
                auto load16 = [&](int cb, uint32_t (&v)[16]) {
                    ptx::tmem_ld_32x32b_x16(tacc + cb * 16, v);
                    ptx::tmem_ld_wait_regs16(v);
#pragma unroll 1
                    for (int jj = 1; jj < n_acc; ++jj) {
                        uint32_t w[16];
                        ptx::tmem_ld_32x32b_x16(tacc + jj * Cfg<V>::ACC_STRIDE + cb * 16, w);
                        ptx::tmem_ld_wait_regs16(w);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            v[i] = __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(w[i]));
                    }
                };
                if (tl.gemm == 1) {
                    // lanes 0..15: gate of unit u, lanes 16..31: up of unit u, u = 64*nb + 16*q + (lane & 15)
                    const int64_t unit = int64_t(tl.nb) * 64 + q * 16 + (lane & 15);
                    uint16_t* h = static_cast<uint16_t*>(p.out);
#pragma unroll 1
                    for (int cb = 0; cb < n_chunks; ++cb) {
                        uint32_t v[16];
                        load16(cb, v);
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
                    if (p.fused) {
                        // publish this warp's part of the segment's h for the GEMM 2 tiles (release at GPU scope)
                        __syncwarp();
                        if (lane == 0) {
                            __threadfence();
                            atomicAdd(&p.seg_done[tl.seg], 1);
                        }
                    }
                } else {
                    void* yout = p.fused ? p.out2 : p.out;
                    const int ydt = p.fused ? p.out2_dtype : p.out_dtype;
                    const int64_t col = int64_t(tl.nb) * 128 + q * 32 + lane;   // output hidden index
#pragma unroll 1
                    for (int cb = 0; cb < n_chunks; ++cb) {
                        uint32_t v[16];
                        load16(cb, v);
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
                            if (ydt == MOE_BF16)
                                static_cast<uint16_t*>(yout)[dst_row * p.K + col] = float_to_bf16_bits(val);
                            else
                                static_cast<float*>(yout)[dst_row * p.K + col] = val;
                        }
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

// ---- host: tensor maps -------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

int make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
             const cuuint32_t* box, const char* what, bool bytes = false) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(MOE_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    // every tile lands 128-byte swizzled: bf16 operands for the MMA, E4M3 code rows (128 bytes) for the
    // converters' conflict-free reads
    CUresult r = fn(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cuuint32_t(rank),
                    const_cast<void*>(base), dims, strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(MOE_ERR_ALIGNMENT, std::string("cuTensorMapEncodeTiled failed for ") + what + " (CUresult " +
                                           std::to_string(int(r)) + ")");
    return MOE_OK;
}


// Tensor maps depend only on pointers and shapes, which repeat call after call:
// they are encoded once and kept (up to 256 shapes; the cache is cleared when full).
struct MapKey {
    int dev;
    const void* a;
    const void* w;
    int64_t kdim, rows_cap, wrows, I, K;
    int E, gemm, swap, w_mode;
    bool operator==(const MapKey& o) const {
        return dev == o.dev && a == o.a && w == o.w && kdim == o.kdim && rows_cap == o.rows_cap && wrows == o.wrows && I == o.I &&
               K == o.K && E == o.E && gemm == o.gemm && swap == o.swap && w_mode == o.w_mode;
    }
};

struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        size_t h = std::hash<const void*>()(k.a) * 31 + std::hash<const void*>()(k.w);
        h = h * 31 + std::hash<int64_t>()(k.kdim * 1000003 + k.rows_cap);
        h = h * 31 + std::hash<int64_t>()(k.wrows * 7 + k.I * 13 + k.K * 17 + k.E);
        return h * 31 + size_t(k.gemm * 8 + k.swap * 4 + k.w_mode + k.dev * 64);
    }
};

std::mutex g_map_mu;
std::unordered_map<MapKey, MapSet, MapKeyHash> g_maps;

}  // namespace

// Test hook for the bounded waits: when the environment variable MOE_TEST_SKIP_FIRST_COPY is 1 at the
// first launch, CTA 0 of every tcgen05 GEMM announces its first stage's bytes but never issues the copy,
// so that stage's "full" barrier never completes.  The MMA issuer's wait then runs out after 2 s, the
// kernel records MOE_DEVERR_TIMEOUT and returns; nothing faults or hangs.  Off unless set.
bool timeout_test_hook() {
    static const bool on = [] {
        const char* v = std::getenv("MOE_TEST_SKIP_FIRST_COPY");
        return v && v[0] == '1';
    }();
    return on;
}

template <int V>
int set_smem_attr() {
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && !done[dev]) {
        if (cudaFuncSetAttribute(gemm_tc_kernel<V>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<V>::SMEM) !=
            cudaSuccess)
            return fail(MOE_ERR_LAUNCH, "cudaFuncSetAttribute(max dynamic smem) failed");
        done[dev] = true;
    }
    return MOE_OK;
}

// Tensor maps of one tile kind: activation rows (128 per normal tile, 16-row boxes for swap-AB) and
// weight rows (256 per normal tile, 128 per swap-AB tile; E4M3 codes as plain bytes).
int build_maps(const GemmArgs& g, bool swap, bool w8, int64_t kdim, int64_t wrows, CUtensorMap* act,
               CUtensorMap* w) {
    const int wtile = swap ? 128 : 256;
    {
        cuuint64_t dims[2] = {cuuint64_t(kdim), cuuint64_t(g.rows_cap)};
        cuuint64_t str[1] = {cuuint64_t(kdim * 2)};
        cuuint32_t box[2] = {BK, cuuint32_t(swap ? TOK_BOX : BM)};
        int rc = make_map(act, g.a, 2, dims, str, box, "activations");
        if (rc) return rc;
    }
    const int64_t es = w8 ? 1 : 2;
    const cuuint32_t kbox = cuuint32_t(w8 ? BK * Cfg<V_E4M3>::KSUB : BK);
    if (g.w1_layout == MOE_W_TILED) {
        // tile-contiguous weights (moe_tile_weights): [E x 128-row blocks][k-blocks][128 rows][128 bytes] (64 bf16
        // or 128 E4M3 codes per row piece, one 16 KB block per stage)
        const cuuint64_t kb = cuuint64_t(128 / es);
        cuuint64_t dims[4] = {kb, 128, cuuint64_t(kdim) / kb, cuuint64_t(g.E * (wrows / 128))};
        cuuint64_t str[3] = {128, 128 * 128, cuuint64_t(kdim) / kb * 128 * 128};
        cuuint32_t box[4] = {cuuint32_t(kb), 128, 1, 1};
        return make_map(w, g.w, 4, dims, str, box, g.gemm == 1 ? "W1 (tiled)" : "W2 (tiled)", w8);
    }
    if (g.gemm == 1 && g.w1_layout == MOE_W1_GATE_UP) {
        // view W1[e] (2I, K) as (K, 16, 2, I/16): row = half*I + 16*blk + q
        cuuint64_t dims[5] = {cuuint64_t(g.K), 16, 2, cuuint64_t(g.I / 16), cuuint64_t(g.E)};
        cuuint64_t str[4] = {cuuint64_t(g.K * es), cuuint64_t(g.I * g.K * es), cuuint64_t(16 * g.K * es),
                             cuuint64_t(2 * g.I * g.K * es)};
        cuuint32_t box[5] = {kbox, 16, 2, cuuint32_t(wtile / 32), 1};
        return make_map(w, g.w, 5, dims, str, box, "W1 (gate/up view)", w8);
    }
    cuuint64_t dims[3] = {cuuint64_t(kdim), cuuint64_t(wrows), cuuint64_t(g.E)};
    cuuint64_t str[2] = {cuuint64_t(kdim * es), cuuint64_t(wrows * kdim * es)};
    cuuint32_t box[3] = {kbox, cuuint32_t(wtile), 1};
    return make_map(w, g.w, 3, dims, str, box, g.gemm == 1 ? "W1" : "W2", w8);
}

// Tensor maps of one launch (normal or swap-AB tiles, and for mixed launches both), encoded once per shape.
int cached_maps(const GemmArgs& g, int mode, bool w8, int64_t kdim, int64_t wrows, int w_mode, MapSet* out) {
    const bool swap = mode == TC_SWAP, mixed = mode == TC_MIXED;
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    const MapKey key{dev_id, g.a, g.w, kdim, g.rows_cap, wrows, g.I, g.K, g.E, g.gemm,
                     mode | (w8 ? 4 : 0), w_mode};
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        auto it = g_maps.find(key);
        if (it != g_maps.end()) {
            *out = it->second;
            return MOE_OK;
        }
    }
    MapSet maps;
    int rc = build_maps(g, swap, w8, kdim, wrows, &maps.act, &maps.w);
    if (rc) return rc;
    if (mixed) {
        rc = build_maps(g, true, w8, kdim, wrows, &maps.act_s, &maps.w_s);
        if (rc) return rc;
    } else {
        maps.act_s = maps.act;
        maps.w_s = maps.w;
    }
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (g_maps.size() >= 256) g_maps.clear();
    g_maps[key] = maps;
    *out = maps;
    return MOE_OK;
}

int launch_gemm_tc(const GemmArgs& g, int mode, cudaStream_t s) {
    const bool swap = mode == TC_SWAP, mixed = mode == TC_MIXED;
    const bool w8 = g.w_dtype == MOE_E4M3;
    if (g.a_dtype != MOE_BF16 || (g.w_dtype != MOE_BF16 && !w8))
        return fail(MOE_ERR_UNSUPPORTED, "tcgen05 path: bf16 activations with bf16 or E4M3 weights only");
    if (w8 && !swap) return fail(MOE_ERR_UNSUPPORTED, "tcgen05 path: E4M3 weights run on swap-AB tiles only");
    if (w8 && !g.w_scale) return fail(MOE_ERR_INVALID_ARG, "tcgen05 path: E4M3 weights need scales");
    if (g.gemm == 1 && g.out_dtype != MOE_BF16) return fail(MOE_ERR_UNSUPPORTED, "tcgen05 GEMM 1 writes bf16 h");
    const int64_t kdim = g.gemm == 1 ? g.K : g.I;
    if (kdim % BK != 0) return fail(MOE_ERR_UNSUPPORTED, "tcgen05 path: contraction length must be a multiple of 64");
    if (w8 && kdim % (BK * Cfg<V_E4M3>::KSUB) != 0)
        return fail(MOE_ERR_UNSUPPORTED, "tcgen05 path: E4M3 weights need a contraction length multiple of 128");
    const int64_t wrows = g.gemm == 1 ? 2 * g.I : g.K;   // weight rows per expert
    const int wtile = swap ? 128 : 256;
    if (wrows % wtile != 0)
        return fail(MOE_ERR_UNSUPPORTED, "tcgen05 path: weight rows per expert must be a multiple of the tile");
    if (g.gemm == 1 && g.w1_layout == MOE_W1_GATE_UP && g.I % 16 != 0)
        return fail(MOE_ERR_UNSUPPORTED, "tcgen05 path: I must be a multiple of 16");
    if (g.rows_cap >= (int64_t(1) << 31)) return fail(MOE_ERR_UNSUPPORTED, "tcgen05 path: too many rows");
    if (g.rows_cap == 0) return MOE_OK;   // no rows, nothing to do

    const int w_mode = g.w1_layout == MOE_W_TILED ? 2 : ((g.gemm == 1 && g.w1_layout == MOE_W1_GATE_UP) ? 1 : 0);
    MapSet maps;
    int rc0 = cached_maps(g, mode, w8, kdim, wrows, w_mode, &maps);
    if (rc0) return rc0;

    TcParams p{};
    p.gemm = g.gemm;
    p.swap = swap ? 1 : 0;
    p.layout = g.layout;
    p.E = g.E;
    p.max_tokens = g.max_tokens;
    p.rows_cap = g.rows_cap;
    p.nkb = int(kdim / (BK * (w8 ? Cfg<V_E4M3>::KSUB : 1)));   // stages per tile
    p.nt = int(wrows / wtile);
    p.mixed = mixed ? 1 : 0;
    p.nt_n = int(wrows / 256);
    p.nt_s = int(wrows / 128);
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
    // bf16 swap-AB launches use the narrow 8-stage ring (64-token spans).  Normal tiles of the batched layout
    // are 256 rows, so one tile covers an expert of up to max_tokens = 256 and streams each weight tile once;
    // the contiguous layout keeps 128-row tiles, whose second accumulator hides the epilogue (measured on the
    // skewed prefill: 256-row tiles took GEMM 1 from 0.629 to 0.665 ms)
    // E4M3 weights: 32-token tiles with four MMA warps when the routed rows average 16 or fewer per expert (the
    // decode regime; an expert with more tokens takes several tiles), else 64-token tiles with two
    const int64_t rows_all = g.layout == MOE_LAYOUT_CONTIGUOUS ? g.rows_cap : int64_t(g.E) * g.max_tokens;
    const int variant = w8 ? (rows_all <= 16 * int64_t(g.E) ? V_E4M3N : V_E4M3)
                           : (swap ? V_SWAP64
                                   : ((mixed || g.layout == MOE_LAYOUT_CONTIGUOUS) ? V_BF16 : V_WIDE));
    p.span = swap ? (variant == V_E4M3    ? Cfg<V_E4M3>::TOK_SPAN
                     : variant == V_E4M3N ? Cfg<V_E4M3N>::TOK_SPAN
                                          : Cfg<V_SWAP64>::TOK_SPAN)
                  : (variant == V_WIDE ? 2 * BM : BM);
    p.w_scale = g.w_scale;
    p.act = static_cast<const uint16_t*>(g.a);
    p.act_ld = kdim;
    p.wrows = wrows;
    p.nsb = kdim / 32;
    p.skip_first_copy = timeout_test_hook() ? 1 : 0;

    int rc = variant == V_E4M3     ? set_smem_attr<V_E4M3>()
             : variant == V_E4M3N  ? set_smem_attr<V_E4M3N>()
             : variant == V_SWAP64 ? set_smem_attr<V_SWAP64>()
             : variant == V_WIDE   ? set_smem_attr<V_WIDE>()
                                   : set_smem_attr<V_BF16>();
    if (rc) return rc;
    // upper bound on the tiles, then one CTA per SM at most
    const int span = p.span;
    int64_t segs;
    if (g.layout == MOE_LAYOUT_CONTIGUOUS) segs = (g.rows_cap + span - 1) / span + g.E;
    else segs = int64_t(g.E) * ((g.max_tokens + span - 1) / span);
    const int64_t tiles = segs * p.nt + (mixed ? int64_t(g.E) * p.nt_s : 0);
    if (tiles == 0) return MOE_OK;
    const int grid = int(std::min<int64_t>(tiles, num_sms()));
    if (variant == V_E4M3)
        gemm_tc_kernel<V_E4M3><<<grid, Cfg<V_E4M3>::THREADS, Cfg<V_E4M3>::SMEM, s>>>(maps.act, maps.w, maps.act_s,
                                                                                     maps.w_s, p);
    else if (variant == V_E4M3N)
        gemm_tc_kernel<V_E4M3N><<<grid, Cfg<V_E4M3N>::THREADS, Cfg<V_E4M3N>::SMEM, s>>>(
            maps.act, maps.w, maps.act_s, maps.w_s, p);
    else if (variant == V_SWAP64)
        gemm_tc_kernel<V_SWAP64><<<grid, Cfg<V_SWAP64>::THREADS, Cfg<V_SWAP64>::SMEM, s>>>(
            maps.act, maps.w, maps.act_s, maps.w_s, p);
    else if (variant == V_WIDE)
        gemm_tc_kernel<V_WIDE><<<grid, Cfg<V_WIDE>::THREADS, Cfg<V_WIDE>::SMEM, s>>>(maps.act, maps.w, maps.act_s,
                                                                                     maps.w_s, p);
    else
        gemm_tc_kernel<V_BF16><<<grid, Cfg<V_BF16>::THREADS, Cfg<V_BF16>::SMEM, s>>>(maps.act, maps.w, maps.act_s,
                                                                                     maps.w_s, p);
    return check_launch("gemm_tc_kernel");
}

size_t experts_fused_workspace_bytes(int64_t rows_cap, int E) {
    const int64_t segs = (rows_cap + Cfg<V_SWAP64>::TOK_SPAN - 1) / Cfg<V_SWAP64>::TOK_SPAN + E;
    return size_t((segs * 4 + 255) / 256 * 256);
}

// GEMM 1 and GEMM 2 of the bf16 swap-AB regime in one cooperative launch (all CTAs resident, so a GEMM 2 tile
// may wait for the GEMM 1 tiles of its token segment, which other resident CTAs reach first in tile order).
int launch_experts_fused(const GemmArgs& g1, const GemmArgs& g2, int32_t* seg_done, size_t ws_bytes,
                         cudaStream_t s) {
    if (g1.a_dtype != MOE_BF16 || g1.w_dtype != MOE_BF16 || g2.w_dtype != MOE_BF16 || g1.out_dtype != MOE_BF16)
        return fail(MOE_ERR_UNSUPPORTED, "fused experts: bf16 activations, weights and h only");
    if (g1.layout != MOE_LAYOUT_CONTIGUOUS) return fail(MOE_ERR_UNSUPPORTED, "fused experts: contiguous layout only");
    if (g1.K % 128 != 0 || g1.I % 64 != 0)
        return fail(MOE_ERR_UNSUPPORTED, "fused experts: K % 128 == 0 and I % 64 == 0 needed");
    if (g1.rows_cap >= (int64_t(1) << 31)) return fail(MOE_ERR_UNSUPPORTED, "fused experts: too many rows");
    if (ws_bytes < experts_fused_workspace_bytes(g1.rows_cap, g1.E))
        return fail(MOE_ERR_WORKSPACE_TOO_SMALL, "fused experts: workspace smaller than moe_experts_fused_workspace_size()");
    if (g1.rows_cap == 0) return MOE_OK;
    const bool tiled = g1.w1_layout == MOE_W_TILED;
    const int w_mode = tiled ? 2 : (g1.w1_layout == MOE_W1_GATE_UP ? 1 : 0);
    MapSet m1, m2;
    int rc = cached_maps(g1, TC_SWAP, false, g1.K, 2 * g1.I, w_mode, &m1);
    if (rc) return rc;
    rc = cached_maps(g2, TC_SWAP, false, g1.I, g1.K, tiled ? 2 : 0, &m2);
    if (rc) return rc;

    TcParams p{};
    p.gemm = 1;
    p.swap = 1;
    p.layout = MOE_LAYOUT_CONTIGUOUS;
    p.E = g1.E;
    p.rows_cap = g1.rows_cap;
    p.nkb = int(g1.K / BK);
    p.nt = int(2 * g1.I / 128);
    p.w_mode = w_mode;
    p.I = g1.I;
    p.K = g1.K;
    p.counts = g1.counts;
    p.offsets = g1.offsets;
    p.row_route = g2.row_route;
    p.route_w = g2.route_w;
    p.out = g1.out;
    p.out_dtype = MOE_BF16;
    p.out_rows = g2.out_rows;
    p.err_word = g1.err_word;
    p.span = Cfg<V_SWAP64>::TOK_SPAN;
    p.wrows = 2 * g1.I;
    p.fused = 1;
    p.nkb2 = int(g1.I / BK);
    p.nt2 = int(g1.K / 128);
    p.w_mode2 = tiled ? 2 : 0;
    p.out2 = g2.out;
    p.out2_dtype = g2.out_dtype;
    p.seg_done = seg_done;
    p.skip_first_copy = timeout_test_hook() ? 1 : 0;

    rc = set_smem_attr<V_SWAP64>();
    if (rc) return rc;
    const int64_t segs = (g1.rows_cap + p.span - 1) / p.span + g1.E;
    if (cudaMemsetAsync(seg_done, 0, size_t(segs) * 4, s) != cudaSuccess)
        return fail(MOE_ERR_LAUNCH, "fused experts: clearing the segment counters failed");
    const int64_t tiles = segs * (p.nt + p.nt2);
    const int grid = int(std::min<int64_t>(tiles, num_sms()));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(Cfg<V_SWAP64>::THREADS);
    cfg.dynamicSmemBytes = Cfg<V_SWAP64>::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, gemm_tc_kernel<V_SWAP64>, m1.act, m1.w, m2.act, m2.w, p) != cudaSuccess)
        return check_launch("gemm_tc_kernel (fused experts)");
    return check_launch("gemm_tc_kernel (fused experts)");
}

}  // namespace moe
