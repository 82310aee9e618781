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
// Lane l holds the 28 logits with ids 32*j + l.  A threshold T = the 16th
// largest of the 32 lane maxima is a lower bound on the 16th largest key
// (at least 16 lanes hold a key >= T), so only keys >= T can be picked.
// Those candidates (usually a few dozen) are compacted into shared memory and
// each finds its rank among them by counting; ranks 0..15 are the picks.
// Rows with more than 64 candidates (heavy ties) take 16 rounds of
// (largest key, smallest id) warp reductions over all 896 keys instead.
// Both give the unique ranking above.
//
// Weights: w_i = s_i / sum_j s_j, s_i = 1 / (1 + exp(-logit_i)) (the
// library's stated convention), in FP32 with compensated (two-float) steps
// so that the only sizeable error left is that of expf.
#pragma once

#include <cstdint>

namespace route {

constexpr int kExpertsTopk = 896;
constexpr int kPerLane = kExpertsTopk / 32;  // 28 logits per lane; lane l holds ids 32*j + l
constexpr int kCandMax = 64;        // candidate buffer per warp (two per lane)

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

// The 16th largest of the 32 lanes' values (bitonic sort, ascending).
__device__ __forceinline__ uint32_t warp_16th_largest(uint32_t v, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, v, j);
            const bool ascending = (lane & k) == 0 || k == 32;
            const bool lower = (lane & j) == 0;
            v = (lower == ascending) ? min(v, other) : max(v, other);
        }
    }
    return __shfl_sync(0xFFFFFFFFu, v, 16);
}

// A candidate as one 64-bit word: the key above the complemented id, so that
// a larger word ranks first (larger key; on equal keys, the lower id).
__device__ __forceinline__ unsigned long long pack_cand(uint32_t key, uint32_t id) {
    return ((unsigned long long)key << 32) | (unsigned long long)(~id);
}

// Rank the `total` (<= kCandMax) candidates in `cand` (shared memory, packed
// words, final before the call): each candidate's rank is the number of
// candidates that precede it in the ranking; ranks are distinct (ids are), so
// rank < 16 places a pick.  Lane i < 16 returns the i-th pick.  All 32 lanes
// call it.
__device__ __forceinline__ void pick16_from_candidates(uint2 *cand_words, uint32_t total, int lane,
                                                       uint32_t &mine_key, uint32_t &mine_id) {
    unsigned long long *cand = reinterpret_cast<unsigned long long *>(cand_words);
    const bool has0 = (uint32_t)lane < total, has1 = (uint32_t)lane + 32u < total;
    const unsigned long long c0 = has0 ? cand[lane] : 0ull;
    const unsigned long long c1 = has1 ? cand[lane + 32] : 0ull;
    uint32_t rank0 = 0u, rank1 = 0u;
#pragma unroll 4
    for (uint32_t j = 0; j < total; ++j) {
        const unsigned long long o = cand[j];
        rank0 += o > c0 ? 1u : 0u;
        rank1 += o > c1 ? 1u : 0u;
    }
    __syncwarp();
    if (has0 && rank0 < 16u) cand[rank0] = c0;
    if (has1 && rank1 < 16u) cand[rank1] = c1;
    __syncwarp();
    mine_key = 0u;
    mine_id = 0u;
    if (lane < 16) {
        const unsigned long long c = cand[lane];
        mine_key = (uint32_t)(c >> 32);
        mine_id = ~(uint32_t)c;
    }
    __syncwarp();
}

// Rows with more than kCandMax candidates (heavy ties at the threshold, or
// fewer than 16 numbers): 16 rounds of (largest key, lowest id) over every
// key the warp holds (lane l: ids 32 j + l); lane i < 16 gets the i-th pick.
__device__ __forceinline__ void pick16_by_rounds(uint32_t (&key)[kPerLane], int lane,
                                                 uint32_t &mine_key, uint32_t &mine_id) {
    uint32_t best = 0u;
    int best_j = 0;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j)
        if (key[j] > best) {
            best = key[j];
            best_j = j;
        }
#pragma unroll 1
    for (int i = 0; i < 16; ++i) {
        const uint32_t top = __reduce_max_sync(0xFFFFFFFFu, best);
        const uint32_t c = (best == top) ? (uint32_t)(32 * best_j + lane) : 0xFFFFFFFFu;
        const uint32_t pick = __reduce_min_sync(0xFFFFFFFFu, c);
        if (lane == i) {
            mine_key = top;
            mine_id = pick;
        }
        if ((int)(pick & 31u) == lane) {  // the owner removes the pick and rescans
            const int js = (int)(pick >> 5);
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
}

// Inclusive prefix sum over the lanes; the warp total in `total`.
__device__ __forceinline__ uint32_t warp_inclusive_sum(uint32_t x, int lane, uint32_t &total) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, off);
        if (lane >= off) x += y;
    }
    total = __shfl_sync(0xFFFFFFFFu, x, 31);
    return x;
}

// Routing weights of the 16 picks (lane i < 16 holds pick i) and the
// stores.  FP32 only: t = exp(-|v|) by expf (never overflows); 1 + t is kept
// exactly as a two-float (TwoSum), q = 1 / (1 + t) as a two-float (FMA
// residual), s = q (v >= 0) or t * q (v < 0); the 16 s are summed as
// two-floats in a fixed tree order; w = s / S is rounded once.
//
// sigmoid_terms: s of one pick as a two-float (s_hi, s_lo).
__device__ __forceinline__ void sigmoid_terms(uint32_t key, float &s_hi, float &s_lo) {
    const float v = key_to_float(key);
    const float t = expf(-fabsf(v));
    const float d_hi = 1.0f + t;
    const float bp = d_hi - 1.0f;
    const float d_lo = (1.0f - (d_hi - bp)) + (t - bp);
    const float q_hi = 1.0f / d_hi;
    float r = fmaf(-q_hi, d_hi, 1.0f);
    r = fmaf(-q_hi, d_lo, r);
    const float q_lo = q_hi * r;
    if (v >= 0.0f || v != v) {
        s_hi = q_hi;
        s_lo = q_lo;
    } else {  // t * (q_hi + q_lo) as a two-float
        s_hi = t * q_hi;
        s_lo = fmaf(t, q_hi, -s_hi) + t * q_lo;
    }
}

// The fixed-order two-float total of the 16 lanes' terms (lanes 16..31 hold
// zeros), the weights and the stores.  All 32 lanes call it.
__device__ __forceinline__ void weights16_store_terms(float s_hi, float s_lo, uint32_t mine_id,
                                                      int lane, int32_t *ids_out, float *w_out) {
    float tot_hi = s_hi, tot_lo = s_lo;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) {
        const float o_hi = __shfl_down_sync(0xFFFFFFFFu, tot_hi, off);
        const float o_lo = __shfl_down_sync(0xFFFFFFFFu, tot_lo, off);
        const float sum = tot_hi + o_hi;
        const float bp = sum - tot_hi;
        const float e = (tot_hi - (sum - bp)) + (o_hi - bp);
        tot_hi = sum;
        tot_lo = tot_lo + o_lo + e;
    }
    tot_hi = __shfl_sync(0xFFFFFFFFu, tot_hi, 0);  // lane 0 holds the fixed-order total
    tot_lo = __shfl_sync(0xFFFFFFFFu, tot_lo, 0);
    if (lane < 16) {
        const float q0 = s_hi / tot_hi;
        const float res = fmaf(-q0, tot_hi, s_hi) + s_lo - q0 * tot_lo;
        ids_out[lane] = (int32_t)mine_id;
        w_out[lane] = q0 + res / tot_hi;
    }
}

__device__ __forceinline__ void weights16_store(uint32_t mine_key, uint32_t mine_id, int lane,
                                                int32_t *ids_out, float *w_out) {
    float s_hi = 0.f, s_lo = 0.f;
    if (lane < 16) sigmoid_terms(mine_key, s_hi, s_lo);
    weights16_store_terms(s_hi, s_lo, mine_id, lane, ids_out, w_out);
}

// The calling warp selects the row whose 896 logits it holds (lane l: the
// logits of ids 32 j + l) and writes 16 ids and weights.  All 32 lanes must
// call it; `cand` is this warp's shared buffer of kCandMax entries.  The
// threshold T is the 16th largest of the 32 lane maxima, as keys; when T is
// a number, a logit's key is >= T exactly when the logit is >= the number
// (NaN compares false, -0 equals +0), so only the candidates are turned
// into keys.
__device__ __forceinline__ void topk16_warp_vals(const float (&v)[kPerLane], int32_t *ids_out,
                                                 float *w_out, int lane, uint2 *cand) {
    float m = v[0];
#pragma unroll
    for (int j = 1; j < kPerLane; ++j) m = fmaxf(m, v[j]);  // NaN only if all are NaN
    const uint32_t T = warp_16th_largest(rank_key(m), lane);

    uint32_t mine_key = 0u;  // lane i keeps the i-th pick (i < 16)
    uint32_t mine_id = 0u;
    bool done = false;
    if (T > 1u) {  // a number: not NaN
        const float t = key_to_float(T);
        uint32_t cnt = 0u;
#pragma unroll
        for (int j = 0; j < kPerLane; ++j) cnt += (v[j] >= t) ? 1u : 0u;
        uint32_t total;
        const uint32_t incl = warp_inclusive_sum(cnt, lane, total);
        if (total <= (uint32_t)kCandMax) {
            unsigned long long *c64 = reinterpret_cast<unsigned long long *>(cand);
            uint32_t pos = incl - cnt;
#pragma unroll
            for (int j = 0; j < kPerLane; ++j)
                if (v[j] >= t) c64[pos++] = pack_cand(rank_key(v[j]), (uint32_t)(32 * j + lane));
            __syncwarp();
            pick16_from_candidates(cand, total, lane, mine_key, mine_id);
            done = true;
        }
    }
    if (!done) {
        uint32_t key[kPerLane];
#pragma unroll
        for (int j = 0; j < kPerLane; ++j) key[j] = rank_key(v[j]);
        pick16_by_rounds(key, lane, mine_key, mine_id);
    }
    weights16_store(mine_key, mine_id, lane, ids_out, w_out);
}

// The calling warp selects row `row` (896 logits in global or shared memory,
// final before the call) and writes 16 ids and weights.  All 32 lanes must
// call it; `cand` is this warp's shared buffer of kCandMax entries.
__device__ __forceinline__ void topk16_warp(const float *row, int32_t *ids_out, float *w_out,
                                            int lane, uint2 *cand) {
    float v[kPerLane];
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) v[j] = row[32 * j + lane];
    topk16_warp_vals(v, ids_out, w_out, lane, cand);
}

// The 16 picks (lane i < 16 keeps the i-th, as a key and an id) of the n
// logits of `row` (n <= kExpertsTopk; entries past n take the removed key 0,
// which no real logit maps to, so with n >= 16 none is picked), by the same
// threshold, compaction and ranking as topk16_warp.  All 32 lanes call it.
__device__ __forceinline__ void topk16_warp_picks(const float *row, int n, int lane, uint2 *cand,
                                                  uint32_t &mine_key, uint32_t &mine_id) {
    uint32_t key[kPerLane];
#pragma unroll
    for (int j = 0; j < kPerLane; ++j)
        key[j] = 32 * j + lane < n ? rank_key(row[32 * j + lane]) : 0u;
    uint32_t lane_max = 0u;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) lane_max = max(lane_max, key[j]);
    const uint32_t T = max(warp_16th_largest(lane_max, lane), 1u);
    uint32_t cnt = 0u;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) cnt += (key[j] >= T) ? 1u : 0u;
    uint32_t total;
    const uint32_t incl = warp_inclusive_sum(cnt, lane, total);
    mine_key = 0u;
    mine_id = 0u;
    if (total <= (uint32_t)kCandMax) {
        unsigned long long *c64 = reinterpret_cast<unsigned long long *>(cand);
        uint32_t pos = incl - cnt;
#pragma unroll
        for (int j = 0; j < kPerLane; ++j)
            if (key[j] >= T) c64[pos++] = pack_cand(key[j], (uint32_t)(32 * j + lane));
        __syncwarp();
        pick16_from_candidates(cand, total, lane, mine_key, mine_id);
        return;
    }
    pick16_by_rounds(key, lane, mine_key, mine_id);
}

// Shared memory of topk16_block.
struct TopkBlockSmem {
    uint32_t tmax[kExpertsTopk / 4];  // one key maximum per thread
    alignas(16) uint32_t lmax[32];    // maxima of seven threads' maxima
    uint32_t T;
    uint32_t count;
    uint2 cand[kCandMax];
    uint4 pick[16];                   // (key, id, s_hi, s_lo) of the picks in rank order
};

// The same selection by the 224 threads that hold a row, four logits each
// (v[j] with ids id[j]), spread over every thread so that each step is a
// short one:
//  1. the threshold above: each lane of warp 0 takes the maximum of seven
//     threads' maxima (28 logits); T = the 16th largest of those 32, found
//     by counting (a value's rank is the number of values that precede it,
//     equal values ordered by lane);
//  2. candidates >= T are compacted with a shared counter, one atomic per
//     warp (their order is not fixed; the ranking is);
//  3. each candidate's rank is counted by a quad of threads, each comparing
//     it with a quarter of the candidates, the four counts added by
//     shuffles; ranks 0..15 are the picks, whose sigmoid terms the quad
//     computes before storing them in rank order;
//  4. warp 0 sums the terms and stores ids and weights.
// Rows with more than kCandMax candidates fall back to topk16_warp over
// `row`, the same 896 logits in global memory.  Every one of the 224 threads
// calls it; it uses named barrier `bar`.
__device__ __forceinline__ void topk16_block(const float (&v)[4], const int (&id)[4],
                                             const float *row, int tid, int bar,
                                             TopkBlockSmem &sh, int32_t *ids_out,
                                             float *w_out) {
    constexpr int kThreads = kExpertsTopk / 4;  // 224
    constexpr int kQuads = kThreads / 4;        // 56
    static_assert(2 * kQuads >= kCandMax, "two candidates a quad cover the buffer");
    uint32_t key[4];
    uint32_t m = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        key[j] = rank_key(v[j]);
        m = max(m, key[j]);
    }
    sh.tmax[tid] = m;
    if (tid == 0) sh.count = 0u;
    asm volatile("barrier.sync %0, %1;" ::"r"(bar), "n"(kThreads) : "memory");
    const int lane = tid & 31;
    if (tid < 32) {
        uint32_t lm = 0u;
#pragma unroll
        for (int j = 0; j < kThreads / 32; ++j) lm = max(lm, sh.tmax[tid + 32 * j]);
        sh.lmax[lane] = lm;
        __syncwarp();
        uint32_t before = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint4 o = reinterpret_cast<const uint4 *>(sh.lmax)[j];
            const uint32_t ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                before += (ov[e] > lm || (ov[e] == lm && 4 * j + e < lane)) ? 1u : 0u;
        }
        if (before == 15u) sh.T = lm;  // exactly one lane holds rank 15
    }
    asm volatile("barrier.sync %0, %1;" ::"r"(bar), "n"(kThreads) : "memory");
    const uint32_t T = sh.T;
    // Compaction, one shared atomic per warp: a ballot per key slot gives
    // each candidate its place within the warp's share.
    const uint32_t below = (1u << lane) - 1u;
    uint32_t ball[4], wcount = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        ball[j] = __ballot_sync(0xFFFFFFFFu, key[j] >= T);
        wcount += __popc(ball[j]);
    }
    uint32_t base = 0u;
    if (lane == 0 && wcount != 0u) base = atomicAdd(&sh.count, wcount);
    base = __shfl_sync(0xFFFFFFFFu, base, 0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (key[j] >= T) {
            const uint32_t pos = base + __popc(ball[j] & below);
            if (pos < (uint32_t)kCandMax) sh.cand[pos] = make_uint2(key[j], (uint32_t)id[j]);
        }
        base += __popc(ball[j]);
    }
    asm volatile("barrier.sync %0, %1;" ::"r"(bar), "n"(kThreads) : "memory");
    const uint32_t total = sh.count;
    if (total > (uint32_t)kCandMax) {  // the same for every thread
        if (tid < 32) topk16_warp(row, ids_out, w_out, tid, sh.cand);
        return;
    }
    const uint32_t q = (uint32_t)tid >> 2, part = (uint32_t)tid & 3u;
    const bool has0 = q < total, has1 = q + kQuads < total;
    const uint2 c0 = has0 ? sh.cand[q] : make_uint2(0u, 0xFFFFFFFFu);
    const uint2 c1 = has1 ? sh.cand[q + kQuads] : make_uint2(0u, 0xFFFFFFFFu);
    uint32_t rank0 = 0u, rank1 = 0u;
#pragma unroll 4
    for (uint32_t j = part; j < total; j += 4u) {
        const uint2 o = sh.cand[j];
        rank0 += (o.x > c0.x || (o.x == c0.x && o.y < c0.y)) ? 1u : 0u;
        rank1 += (o.x > c1.x || (o.x == c1.x && o.y < c1.y)) ? 1u : 0u;
    }
    rank0 += __shfl_xor_sync(0xFFFFFFFFu, rank0, 1);
    rank1 += __shfl_xor_sync(0xFFFFFFFFu, rank1, 1);
    rank0 += __shfl_xor_sync(0xFFFFFFFFu, rank0, 2);
    rank1 += __shfl_xor_sync(0xFFFFFFFFu, rank1, 2);
    // Parts 0 and 1 of the quad place candidates c0 and c1 (ranks are distinct).
    const bool mine = part == 0u ? has0 && rank0 < 16u : part == 1u && has1 && rank1 < 16u;
    if (mine) {
        const uint2 c = part == 0u ? c0 : c1;
        float s_hi, s_lo;
        sigmoid_terms(c.x, s_hi, s_lo);
        sh.pick[part == 0u ? rank0 : rank1] =
            make_uint4(c.x, c.y, __float_as_uint(s_hi), __float_as_uint(s_lo));
    }
    asm volatile("barrier.sync %0, %1;" ::"r"(bar), "n"(kThreads) : "memory");
    if (tid >= 32) return;
    uint4 p = make_uint4(0u, 0u, 0u, 0u);
    if (lane < 16) p = sh.pick[lane];
    weights16_store_terms(__uint_as_float(p.z), __uint_as_float(p.w), p.y, lane, ids_out, w_out);
}

}  // namespace route
