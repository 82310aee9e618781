// Warp-per-row standalone top-16 over 896 FP32 router logits, with routing
// weights.  Steps a3/a4 of the route step ("Kimi K3.1 recipe: route 9..20
// decode rows through the pushed pair gather and standalone top-16", commit
// message: the standalone top-16 selects each row's experts).
//
// Ranking: larger logit first; equal logits (with -0 == +0) go to the lower
// expert id; NaN ranks below every number.  Each logit is mapped to a 32-bit
// unsigned key whose integer order is that ranking, so a pick is
// (largest key, then smallest id) and needs two warp reductions.
//
// Weights: w_i = s_i / sum_j s_j, s_i = 1 / (1 + exp(-logit_i)), evaluated in
// double and rounded once to FP32 (the library's stated convention).
#pragma once

#include <cstdint>

namespace route {

constexpr int kPerLane = 896 / 32;  // 28 logits per lane; lane l holds ids 32*j + l

// Order-preserving key: NaN -> 1 (below -Inf), -0 -> +0, removed entries -> 0.
__device__ __forceinline__ uint32_t rank_key(float v) {
    uint32_t b = __float_as_uint(v);
    uint32_t mag = b & 0x7FFFFFFFu;
    if (mag > 0x7F800000u) return 1u;
    if (mag == 0u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Inverse of rank_key for keys >= 1 (NaN comes back as a NaN).
__device__ __forceinline__ float key_to_float(uint32_t key) {
    uint32_t b = (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
    return __uint_as_float(b);
}

// The calling warp selects row `row` (896 logits, read through L2 so that
// values written by other CTAs of the same kernel are seen) and writes 16 ids
// and weights.  All 32 lanes must call it.
__device__ __forceinline__ void topk16_warp(const float *row, int32_t *ids_out, float *w_out,
                                            int lane) {
    uint32_t key[kPerLane];
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) key[j] = rank_key(__ldcg(row + 32 * j + lane));

    uint32_t best = 0u;
    int best_j = 0;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j)
        if (key[j] > best) {
            best = key[j];
            best_j = j;
        }

    uint32_t mine_key = 0u;  // lane i keeps the i-th pick (i < 16)
    uint32_t mine_id = 0u;
#pragma unroll 1
    for (int i = 0; i < 16; ++i) {
        uint32_t top = __reduce_max_sync(0xFFFFFFFFu, best);
        uint32_t cand = (best == top) ? (uint32_t)(32 * best_j + lane) : 0xFFFFFFFFu;
        uint32_t pick = __reduce_min_sync(0xFFFFFFFFu, cand);
        if (lane == i) {
            mine_key = top;
            mine_id = pick;
        }
        if ((int)(pick & 31u) == lane) {  // the owner removes the pick and rescans
            int js = (int)(pick >> 5);
            best = 0u;
            best_j = 0;
#pragma unroll
            for (int j = 0; j < kPerLane; ++j) {
                if (j == js) key[j] = 0u;
                if (key[j] > best) {
                    best = key[j];
                    best_j = j;
                }
            }
        }
    }

    double s = 0.0;
    if (lane < 16) s = 1.0 / (1.0 + exp(-(double)key_to_float(mine_key)));
    double total = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) total += __shfl_xor_sync(0xFFFFFFFFu, total, off);
    total = __shfl_sync(0xFFFFFFFFu, total, 0);  // one association order for every lane
    if (lane < 16) {
        ids_out[lane] = (int32_t)mine_id;
        w_out[lane] = (float)(s / total);
    }
}

}  // namespace route
