// Per-token top-k routing, shared by the route kernel and the fused
// route + permute kernel: one warp holds a token's E logits in registers
// (E/32 per lane), takes the top k by repeated warp arg-max with the lower
// index winning ties, and forms softmax weights over the chosen (or all)
// logits.  NaN logits are outside the contract.
#pragma once

#include <float.h>

#include "common.cuh"

namespace moe {
namespace {

// Order-preserving key of a logit: for finite values and +-inf, a > b as
// floats exactly when key(a) > key(b) as unsigned integers.  -0 is folded into
// +0 first (the two compare equal as floats), so equal floats get equal keys.
// Every key is >= 0x007fffff (the key of -inf), so 0 can mark "no candidate";
// key_value inverts the map (returning +0 for either zero).
MOE_DEVICE uint32_t order_key(float v) {
    const uint32_t u = __float_as_uint(v + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

MOE_DEVICE float key_value(uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k); }

// Called by all 32 lanes of a warp for the token whose logits start at `row`.
// Lane j < k receives the j-th chosen expert (decreasing logit, the lower
// index first among equal logits) in *id and its weight in *weight; other
// lanes receive -1 and 0.  Each of the k rounds takes the warp maximum of the
// lanes' best keys and then the lowest expert index holding that key
// (redux.sync).  With at most 8 entries per lane, each lane sorts its entries
// once (stable, decreasing key), so its best is always its first entry and the
// winning lane shifts its list; with more, each round rescans the lane's
// remaining entries.  The weights are formed after the selection: lane j takes
// p_j = exp(l_j - l_max), and the sum of the p_j is accumulated in j order.
template <int PER_LANE>
MOE_DEVICE void route_token(const float* __restrict__ row, int E, int k, int renorm, int lane, int* id,
                            float* weight) {
    constexpr bool kSorted = PER_LANE <= 8;
    uint32_t key[PER_LANE];
    int slot[PER_LANE];   // entry i of this lane is expert i*32 + lane
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
        const int e = i * 32 + lane;
        key[i] = e < E ? order_key(row[e]) : 0u;   // 0: never a candidate
        slot[i] = i;
    }
    // softmax over all E: the sum of exp(l - l_max) in entry order, then across lanes
    float denom_all = 0.f;
    if (!renorm) {
        uint32_t lm = 0u;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) lm = max(lm, key[i]);
        const float lmax0 = key_value(__reduce_max_sync(0xffffffffu, lm));
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i)
            if (i * 32 + lane < E) denom_all += expf(key_value(key[i]) - lmax0);
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) denom_all += __shfl_xor_sync(0xffffffffu, denom_all, d);
    }
    if constexpr (kSorted) {
        // odd-even transposition sort; swapping only strictly smaller keys keeps equal keys in index order
#pragma unroll
        for (int pass = 0; pass < PER_LANE; ++pass) {
#pragma unroll
            for (int i = pass & 1; i + 1 < PER_LANE; i += 2) {
                if (key[i] < key[i + 1]) {
                    const uint32_t tk = key[i];
                    key[i] = key[i + 1];
                    key[i + 1] = tk;
                    const int ts = slot[i];
                    slot[i] = slot[i + 1];
                    slot[i + 1] = ts;
                }
            }
        }
    }
    // unsorted variant: entries not taken yet (bit i: entry i)
    uint32_t avail = PER_LANE == 32 ? 0xffffffffu : (1u << (PER_LANE & 31)) - 1u;
    int my_id = -1;
    uint32_t my_key = 0u, lmax_key = 0u;
    for (int j = 0; j < k; ++j) {
        uint32_t bk;
        int bi;
        if constexpr (kSorted) {
            bk = key[0];
            bi = slot[0] * 32 + lane;
        } else {
            bk = 0u;
            bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < PER_LANE; ++i)
                if (((avail >> i) & 1u) && key[i] > bk) { bk = key[i]; bi = i * 32 + lane; }
        }
        // some entry is left (k <= E), so the maximum is a real key and only lanes holding it compete
        const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
        const int ei = __reduce_min_sync(0xffffffffu, bk == mk ? bi : 0x7fffffff);
        if ((ei & 31) == lane) {
            if constexpr (kSorted) {
#pragma unroll
                for (int i = 0; i + 1 < PER_LANE; ++i) {
                    key[i] = key[i + 1];
                    slot[i] = slot[i + 1];
                }
                key[PER_LANE - 1] = 0u;
            } else {
                avail &= ~(1u << (ei >> 5));
            }
        }
        if (j == 0) lmax_key = mk;
        if (lane == j) { my_id = ei; my_key = mk; }
    }
    const float lmax = key_value(lmax_key);
    const float p = lane < k ? expf(key_value(my_key) - lmax) : 0.f;
    float denom = denom_all;
    if (renorm) {
        for (int j = 0; j < k; ++j) denom += __shfl_sync(0xffffffffu, p, j);
    }
    *id = my_id;
    *weight = lane < k ? p / denom : 0.f;
}

}  // namespace
}  // namespace moe
