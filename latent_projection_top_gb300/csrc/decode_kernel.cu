// Decode route step (1..20 token rows): steps a1..a4 as two kernels.
//
//   latent[r, n] = bf16( sum_k hidden[r, k] * W_latent[k, n] )   n < 3584
//   logits[r, e] =       sum_k hidden[r, k] * W_router[k, e]    e < 896
//   ids / weights = top-16 of logits[r, :]
//
// At decode widths the step is a stream of the 64.2 MB of weights; the
// arithmetic is small.  The kernels are built around that stream.
//
// decode_stream_kernel -- one CTA per SM.  The weights are cut into 18
//   column tiles of 256 columns (14 latent, 4 router; the last router tile
//   has 128 real columns and TMA zero-fills the rest) and 112 k-blocks of 64;
//   CTA g owns a contiguous run of (tile, k-block) units, the same even
//   number for every CTA.  256-column tiles put 512 contiguous bytes per weight
//   row in flight, which the HBM needs to run at full speed.  Per unit a TMA
//   producer brings four 64x64 weight boxes and the hidden box (BN = 16 or 32
//   rows, zero-filled past `rows`) into a 4-stage shared-memory ring; one
//   thread issues tcgen05 MMAs (128 weight columns on M, token rows on N) into
//   a fresh TMEM accumulator per pair of k-blocks (runs are even and tiles
//   start at even units, so a pair never crosses a tile); eight epilogue
//   warps add each pair's FP32 result into a two-float (TwoSum) running sum
//   kept in TMEM next to the accumulators (two rows at a time in packed FP32
//   pairs), so the only rounding left is the tensor core's inside one
//   128-long block.  Pairing halves the epilogue's
//   TMEM traffic, two-float work and barrier hand-offs per streamed byte,
//   which set the pace at 17..20 rows (measured 12.6 -> 11.3 us a layer at
//   20 rows, 10.7 -> 10.4 at 8).  A CTA's run covers at most two tiles; the
//   first run's partial waits in shared memory and both are stored to their
//   scratch slots when the CTA's stream ends.
//
// decode_finish_kernel -- at most one small CTA per SM, so that it fits next
//   to a stream CTA: one CTA per row sums the row's 896 router logits and
//   runs the top-16 on them with all its threads; the others sum the latent
//   tiles, two or four (row, tile) items per memory round trip (or the
//   general path's K-split latent).  Slots are summed in segment order as
//   two-floats and rounded once, so results are bitwise reproducible and a
//   row's bits do not depend on the row count (the partition depends only on
//   the grid).  With each latent row's sum of squares asked for, the same
//   work runs as decode_finish_ss_kernel, one thread-block cluster per row.
//   A column shard's plan streams only its own tiles (up to 64 CTAs a tile)
//   and finishes with decode_shard_finish_kernel, which sums each value's
//   partials with up to four threads and picks the shard's candidates.
//
// Programmatic dependent launch: both kernels let their successor launch at
// once.  The stream kernel requests its first weight boxes (model
// parameters, which no predecessor writes) before `griddepcontrol.wait`, and
// the weights of its next two units into L2, a deeper start than its ring.
// By default it reads the hidden rows only after the wait; with `overlap` set
// it reads them at once and waits only before it writes scratch (at the end
// of its stream), so one step's weight stream runs under the previous step's
// finish kernel.  Rows that a concurrent staging kernel publishes (a host
// step launched behind another step) are read once a device counter says
// they are all there.
#include <cuda_bf16.h>

#include "common.cuh"
#include "sm103_ptx.cuh"
#include "topk16.cuh"
#include "twofloat.cuh"

namespace route {
namespace {

constexpr uint32_t kBoxBytes = 64 * 64 * 2;         // one 64-column x 64-k weight box
constexpr uint32_t kDAStageBytes = 4 * kBoxBytes;   // 256 columns x 64 k
// Warps: 0 TMA producer, 1 MMA issuer, 2..9 epilogue -- warp w drains TMEM
// lanes 32*(w % 4) .. +31 of column block (w - 2) / 4.  The running two-float
// sums stay in TMEM, not registers, so that the small finish CTAs of the
// previous step fit on the same SM.
constexpr int kDecThreads = 320;
constexpr int kEpiThreads = 256;

template <int BN>
struct DecCfg {
    static constexpr uint32_t kBStageBytes = BN * 128;  // BN rows x 64 k, BF16
    static constexpr uint32_t kStageBytes = kDAStageBytes + kBStageBytes;
    static constexpr int kStages = 4;  // measured, with and without the L2 start prefetch: 4 beats 3, 5 and 6
    static constexpr uint32_t kAccCols = 2 * BN;       // two 128-column blocks per accumulator
    // TMEM columns: kNumAcc accumulators (k-block pairs in flight), then the
    // running sums, per column block BN hi columns and BN lo columns.
    static constexpr int kNumAcc = BN == 16 ? 8 : 6;
    static constexpr uint32_t kStateCol = kNumAcc * kAccCols;
    // a CTA's first-run partial waits here until its last run is done, so
    // global scratch is written only at the end of the CTA's stream
    static constexpr uint32_t kStashBytes = kDecodeMaxRows * kDTileCols * 8;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kSmemBytes = 1024 + kStages * kStageBytes + kStashBytes + 256;
    // tcgen05 kind::f16: FP32 accumulator, BF16 A (MN-major) and B (K-major),
    // N = BN token rows, M = 128 weight columns.
    static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) |
                                       ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    static_assert(BN == 16 || BN == 32, "decode row tile");
    static_assert(kDecodeMaxRows > 16 && kDecodeMaxRows - 16 == 4, "BN = 32 drains rows 16..19");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
    static_assert(kStateCol + 4 * BN <= kTmemCols, "TMEM");
};

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;  // descriptor version for tcgen05
    d |= 2ull << 61;  // 128-byte swizzle
    return d;
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// One chunk of W rows (TMEM columns r0 .. r0+W-1) of the epilogue: add the
// k-block pair's result at `acc` into the running two-float sums at s_hi /
// s_lo (or start them, on the first pair of a run); at the end of a run store
// the sums for rows < `rows` to `out` instead.  `release` frees the
// accumulator once its columns are in registers.
template <int W>
__device__ __forceinline__ void epi_chunk(uint32_t acc, uint32_t s_hi, uint32_t s_lo, int r0,
                                          bool run_start, bool run_end, bool release,
                                          uint32_t accempty, float2 *out, int col, int rows) {
    uint32_t v[W], h[W], l[W];
    ptx::tmem_ld(acc + r0, v);
    if (!run_start) {
        ptx::tmem_ld(s_hi + r0, h);
        ptx::tmem_ld(s_lo + r0, l);
    }
    ptx::tmem_ld_wait();
    if (release) {  // the accumulator is free for the next pair
        ptx::tc_fence_before();
        ptx::mbar_arrive(accempty);
    }
    // two rows at a time, in packed FP32 pairs
    static_assert(W % 2 == 0, "rows in pairs");
#pragma unroll
    for (int j = 0; j < W; j += 2) {
        if (run_start) {
            h[j] = v[j];
            h[j + 1] = v[j + 1];
            l[j] = l[j + 1] = 0u;
        } else {
            uint64_t hp = ptx::f32x2_pack(__uint_as_float(h[j]), __uint_as_float(h[j + 1]));
            uint64_t lp = ptx::f32x2_pack(__uint_as_float(l[j]), __uint_as_float(l[j + 1]));
            two_sum_acc_x2(hp, lp,
                           ptx::f32x2_pack(__uint_as_float(v[j]), __uint_as_float(v[j + 1])));
            float a, b;
            ptx::f32x2_unpack(hp, a, b);
            h[j] = __float_as_uint(a);
            h[j + 1] = __float_as_uint(b);
            ptx::f32x2_unpack(lp, a, b);
            l[j] = __float_as_uint(a);
            l[j + 1] = __float_as_uint(b);
        }
    }
    if (!run_end) {
        ptx::tmem_st(s_hi + r0, h);
        ptx::tmem_st(s_lo + r0, l);
    } else {
        // The run's partial: the first of two runs waits in shared memory
        // (each thread reads back only its own entries).
#pragma unroll
        for (int j = 0; j < W; ++j)
            if (r0 + j < rows)
                out[(r0 + j) * kDTileCols + col] =
                    make_float2(__uint_as_float(h[j]), __uint_as_float(l[j]));
    }
}

__device__ __forceinline__ void fail_timeout(const DecodeArgs &a, volatile int *abort_flag) {
    *abort_flag = 1;
    atomicOr(&a.words[kWordStatus], kStatusTimeout);
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const DecodeArgs &a,
                                           volatile int *abort_flag) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0u) {
            if (*abort_flag) return false;
            if (ptx::global_timer_ns() - t0 > a.timeout_ns) {
                fail_timeout(a, abort_flag);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, const DecodeArgs &a) {
    const uint64_t t0 = ptx::global_timer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::global_timer_ns() - t0 > a.timeout_ns) {
            atomicOr(&a.words[kWordStatus], kStatusTimeout);
            return;
        }
    }
}

// Rows published by a concurrent staging kernel (a host step launched behind
// another step): wait until its CTAs have all published them (bounded: after
// the timeout the status word records it and the stream goes on, its
// outputs invalid), then order the acquire before this thread's TMA reads.
__device__ __noinline__ void wait_published(const DecodeArgs &a) {
    const uint64_t t0 = ptx::global_timer_ns();
    while ((int)(ptx::ld_acquire_gpu(a.hidden_count) - a.hidden_target) < 0) {
        if (ptx::global_timer_ns() - t0 > a.timeout_ns) {
            atomicOr(&a.words[kWordStatus], kStatusTimeout);
            break;
        }
    }
    ptx::fence_proxy_async_global();
}

// Register caps (the most each variant compiles to without spilling) leave
// room on every SM sub-partition for two warps of a finish CTA.
template <int BN>
__global__ void __maxnreg__(BN == 16 ? 80 : 88)
    decode_stream_kernel(const __grid_constant__ CUtensorMap map_h,
                         const __grid_constant__ CUtensorMap map_wl,
                         const __grid_constant__ CUtensorMap map_wr,
                         const __grid_constant__ DecodeArgs args) {
    using C = DecCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem_base;
    __shared__ volatile int s_abort;

    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    float2 *const stash =
        reinterpret_cast<float2 *>(smem_raw + (sbase - raw) + C::kStages * C::kStageBytes);
    const uint32_t bars = sbase + C::kStages * C::kStageBytes + C::kStashBytes;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (C::kStages + s); };
    auto accfull_bar = [&](int b) { return bars + 8u * (2 * C::kStages + b); };
    auto accempty_bar = [&](int b) { return bars + 8u * (2 * C::kStages + C::kNumAcc + b); };
    const uint32_t drain_bar = bars + 8u * (2 * C::kStages + 2 * C::kNumAcc);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = blockIdx.x;
    const int u0 = args.cta_unit[g];
    const int u1 = args.cta_unit[g + 1];
    const int n_units = u1 - u0;

    if (threadIdx.x == 0) {
        // Let the next kernel on the stream launch as soon as SMs free up.
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        s_abort = 0;
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < C::kNumAcc; ++b) {
            ptx::mbar_init(accfull_bar(b), 1);
            ptx::mbar_init(accempty_bar(b), kEpiThreads);
        }
        ptx::mbar_init(drain_bar, 1);
        ptx::fence_barrier_init();
        ptx::prefetch_tensormap(&map_h);
        ptx::prefetch_tensormap(&map_wl);
        ptx::prefetch_tensormap(&map_wr);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(&s_tmem_base), C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = s_tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            const uint64_t pol_w = ptx::policy_evict_first();
            const uint64_t pol_h = ptx::policy_evict_last();
            const int n_pre = n_units < C::kStages ? n_units : C::kStages;
            auto weights_of = [&](int u, uint32_t a, uint32_t bar) {
                const int t = u / kKBlocks, kb = u % kKBlocks;
                const bool lat = t < args.lat_tiles;
                const CUtensorMap *wmap = lat ? &map_wl : &map_wr;
                const int x0 = (lat ? t : t - args.lat_tiles) * kDTileCols;
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    ptx::tma_load_2d(a + b * kBoxBytes, wmap, bar, x0 + 64 * b, kb * kKBlock, pol_w);
            };
            uint32_t armed = 0u, armed_par = 0u;
            // Weight boxes of the first stages go out before the grid
            // dependency resolves (no predecessor writes the weights).
            for (int i = 0; i < n_pre; ++i) {
                ptx::mbar_arrive_expect_tx(full_bar(i), C::kStageBytes);
                weights_of(u0 + i, sbase + i * C::kStageBytes, full_bar(i));
                armed |= 1u << i;
            }
            // The next units' weights go to L2 behind them, a deeper start
            // than the ring alone: HBM keeps working while a new CTA's first
            // stages drain (and, without overlap, while the ring waits for
            // the hidden rows once the dependency resolves).  With overlap
            // they are asked for after the first hidden boxes, which the
            // first MMAs need (measured: 0.1-0.25 us a layer at 16-20 rows).
            const int n_l2 = n_units - n_pre < args.pre_l2 ? n_units - n_pre : args.pre_l2;
            auto prefetch_l2 = [&]() {
                for (int i = n_pre; i < n_pre + n_l2; ++i) {
                    const int u = u0 + i, t = u / kKBlocks, kb = u % kKBlocks;
                    const bool lat = t < args.lat_tiles;
                    const int x0 = (lat ? t : t - args.lat_tiles) * kDTileCols;
#pragma unroll
                    for (int b = 0; b < 4; ++b)
                        ptx::tma_prefetch_l2_2d(lat ? &map_wl : &map_wr, x0 + 64 * b, kb * kKBlock);
                }
            };
            if (!args.overlap) {
                prefetch_l2();
                asm volatile("griddepcontrol.wait;" ::: "memory");
            } else if (args.hidden_count != nullptr) {
                wait_published(args);
            }
            for (int i = 0; i < n_pre; ++i) {
                if (args.test_stall && i == n_units - 1) continue;  // test hook
                ptx::tma_load_2d(sbase + i * C::kStageBytes + kDAStageBytes, &map_h, full_bar(i),
                                 ((u0 + i) % kKBlocks) * kKBlock, 0, pol_h);
            }
            if (args.overlap) prefetch_l2();
            bool ok = true;
            for (int i = n_pre; i < n_units; ++i) {
                const int s = i % C::kStages;
                const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
                if (!wait_phase(empty_bar(s), ph ^ 1u, args, &s_abort)) {
                    ok = false;
                    break;
                }
                if (args.test_stall && i == n_units - 1) continue;  // test hook: never filled
                const uint32_t a = sbase + s * C::kStageBytes;
                ptx::mbar_arrive_expect_tx(full_bar(s), C::kStageBytes);
                weights_of(u0 + i, a, full_bar(s));
                ptx::tma_load_2d(a + kDAStageBytes, &map_h, full_bar(s), ((u0 + i) % kKBlocks) * kKBlock,
                                 0, pol_h);
                armed |= 1u << s;
                armed_par = (armed_par & ~(1u << s)) | (ph << s);
            }
            if (!ok || s_abort) {  // let every issued copy land before the CTA may exit
                for (int s = 0; s < C::kStages; ++s)
                    if (armed & (1u << s)) wait_drain(full_bar(s), (armed_par >> s) & 1u, args);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer: one fresh accumulator per k-block pair ----------------
            for (int i = 0; i < n_units; ++i) {
                const int s = i % C::kStages;
                const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
                const int buf = (i >> 1) % C::kNumAcc;
                const uint32_t use = (uint32_t)((i >> 1) / C::kNumAcc);
                if (!(i & 1) && !wait_phase(accempty_bar(buf), (use & 1u) ^ 1u, args, &s_abort))
                    break;
                if (!wait_phase(full_bar(s), ph, args, &s_abort)) break;
                ptx::tc_fence_after();
                const uint32_t a = sbase + s * C::kStageBytes;
                const uint32_t b = a + kDAStageBytes;
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    const uint32_t d_tmem = tmem_base + (uint32_t)(buf * C::kAccCols + blk * BN);
#pragma unroll
                    for (int kk = 0; kk < kKBlock / 16; ++kk) {
                        // A: block blk is boxes 2blk, 2blk+1 (8192 B apart, LBO);
                        //    k advances 16 rows = two 1024-B swizzle atoms (SBO 1024).
                        // B: k advances 32 B within the 128-B swizzled row.
                        const uint64_t da =
                            smem_desc(a + blk * 2 * kBoxBytes + kk * 2048u, kBoxBytes, 1024u);
                        const uint64_t db = smem_desc(b + kk * 32u, 16u, 1024u);
                        ptx::mma_bf16(d_tmem, da, db, C::kIdesc, kk > 0 || (i & 1) ? 1u : 0u);
                    }
                }
                ptx::mma_commit(empty_bar(s));
                if (i & 1) ptx::mma_commit(accfull_bar(buf));
            }
            ptx::mma_commit(drain_bar);  // every MMA retired before TMEM is freed
            wait_drain(drain_bar, 0u, args);
        }
    } else {
        // ---------------- epilogue: two-float sums of the k-block pairs' results ----------------
        const int quarter = warp & 3;        // TMEM lanes 32*quarter .. +31
        const int blk = (warp - 2) >> 2;     // column block 0 or 1 of the tile
        const int col = blk * 128 + 32 * quarter + lane;
        const int rows = args.rows;
        const uint32_t lanes = tmem_base + ((uint32_t)(32 * quarter) << 16);
        const uint32_t sum_hi = lanes + C::kStateCol + (uint32_t)(blk * 2 * BN);
        const uint32_t sum_lo = sum_hi + BN;
        int first_slot = -1;
        bool run_start = true;
        for (int i = 1; i < n_units; i += 2) {  // the second k-block of each pair
            const int u = u0 + i;
            const int t = u / kKBlocks;
            const int buf = (i >> 1) % C::kNumAcc;
            const uint32_t use = (uint32_t)((i >> 1) / C::kNumAcc);
            // Each warp waits on its own; an abort seen by one is seen by all.
            if (!wait_phase(accfull_bar(buf), use & 1u, args, &s_abort)) break;
            __syncwarp();  // the TMEM loads below are warp-wide (.sync.aligned)
            ptx::tc_fence_after();
            const bool last = i == n_units - 1;
            const bool run_end = last || (u + 1) % kKBlocks == 0;
            // Scratch may still be read by the predecessor's finish kernel.
            if (last) asm volatile("griddepcontrol.wait;" ::: "memory");
            const int slot = args.seg_base[t] + (g - args.cta_first[t]);
            [[maybe_unused]] const int nslots =  // read by the checked library's index check
                args.seg_base[args.tiles - 1] + args.seg_count[args.tiles - 1];
            const bool slot_ok = ROUTE_IN_BOUNDS(
                t < args.tiles && slot >= 0 && slot < nslots && col < kDTileCols, args.words);
            float2 *const out =
                last && slot_ok ? args.ws + (size_t)slot * kDecodeMaxRows * kDTileCols : stash;
            const uint32_t acc = lanes + (uint32_t)(buf * C::kAccCols + blk * BN);
            // Rows 0..15, then (BN = 32) rows 16..19: no row past the
            // 20-row envelope is ever read from TMEM.
            epi_chunk<16>(acc, sum_hi, sum_lo, 0, run_start, run_end, BN == 16,
                          accempty_bar(buf), out, col, rows);
            if constexpr (BN == 32)
                epi_chunk<kDecodeMaxRows - 16>(acc, sum_hi, sum_lo, 16, run_start, run_end, true,
                                               accempty_bar(buf), out, col, rows);
            if (!run_end) ptx::tmem_st_wait();  // the next pair reads these sums back
            if (run_end && !last) first_slot = slot;
            if (last && first_slot >= 0 && ROUTE_IN_BOUNDS(first_slot < nslots, args.words)) {
                float2 *p0 = args.ws + (size_t)first_slot * kDecodeMaxRows * kDTileCols;
                for (int r = 0; r < rows; ++r) p0[r * kDTileCols + col] = stash[r * kDTileCols + col];
            }
            run_start = run_end;
        }
        // Every kernel of the chain waits for its predecessor before it ends.
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

// Split-K sums.  A thread sums NP column pairs of one row, each over its
// tile's partial slots in slot order, as two-floats rounded once at the end.
// All slots of all NP pairs are loaded before any is added (one memory round
// trip for up to kFinishBatch slots), at immediate offsets from one pointer
// per pair.
constexpr int kFinishBatch = 10;
constexpr int kSlotF4 = kDecodeMaxRows * kDTileCols / 2;  // float4 (two columns) per slot

// Where the partials of one (row, column pair) sit: the first slot's float4
// and the slot count.  Built from the launch parameters before the grid
// dependency resolves, so that the sums start with the slot loads.
struct SlotRun {
    const float4 *p;
    int n;
};

__device__ __forceinline__ SlotRun slot_run(const DecodeArgs &a, int r, int t, int cc) {
    SlotRun s;
    if (!ROUTE_IN_BOUNDS(r >= 0 && r < a.rows && t >= 0 && t < a.tiles && cc >= 0 &&
                             cc + 1 < kDTileCols,
                         a.words))
        return SlotRun{reinterpret_cast<const float4 *>(a.ws), 0};
    s.p = reinterpret_cast<const float4 *>(a.ws) +
          ((size_t)a.seg_base[t] * kDecodeMaxRows + r) * (kDTileCols / 2) + cc / 2;
    s.n = a.seg_count[t];
    return s;
}

// Keeps `s` computed here: an empty volatile asm is not moved across the
// volatile `griddepcontrol.wait` that follows it.
__device__ __forceinline__ void pin(SlotRun &s) {
    asm volatile("" : "+l"(s.p), "+r"(s.n));
}

template <int NP, int B = kFinishBatch>
__device__ __forceinline__ void sum_slot_pairs(const SlotRun (&run)[NP], float2 (&y)[NP]) {
    const float4 *p[NP];
    int n[NP], nmax = 0;
    float h[2 * NP], l[2 * NP];
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        p[q] = run[q].p;
        n[q] = run[q].n;
        nmax = n[q] > nmax ? n[q] : nmax;
        h[2 * q] = h[2 * q + 1] = l[2 * q] = l[2 * q + 1] = 0.f;
    }
    for (int s0 = 0; s0 < nmax; s0 += B) {
        float4 v[NP][B];
#pragma unroll
        for (int j = 0; j < B; ++j)
#pragma unroll
            for (int q = 0; q < NP; ++q)
                if (s0 + j < n[q]) v[q][j] = __ldcg(p[q] + j * kSlotF4);
#pragma unroll
        for (int j = 0; j < B; ++j)
#pragma unroll
            for (int q = 0; q < NP; ++q)
                if (s0 + j < n[q]) {
                    two_sum_acc(h[2 * q], l[2 * q], v[q][j].x);
                    l[2 * q] += v[q][j].y;
                    two_sum_acc(h[2 * q + 1], l[2 * q + 1], v[q][j].z);
                    l[2 * q + 1] += v[q][j].w;
                }
#pragma unroll
        for (int q = 0; q < NP; ++q) p[q] += B * kSlotF4;
    }
#pragma unroll
    for (int q = 0; q < NP; ++q) y[q] = make_float2(two_float_value(h[2 * q], l[2 * q]),
                                                    two_float_value(h[2 * q + 1], l[2 * q + 1]));
}

// The general path's latent arithmetic ("Optionally gather the Kimi3 prefill
// latent instead of reducing it", Description, Numerics bullet, and commit
// body: eight K-slice partials, each rounded to BF16, summed in FP32, rounded
// to BF16 again).  With the partition aligned to the eight 896-deep K slices
// (checked on the host), slot j of a latent tile is slice j: each slot's
// two-float partial is rounded to FP32 and then to BF16, and the BF16 values
// are added in FP32 in slice order; the caller rounds the sum to BF16.
// NP column pairs at a time, all their slots loaded before any is added.
template <int NP>
__device__ __forceinline__ void ksplit_slot_pairs(const SlotRun (&run)[NP], float2 (&y)[NP]) {
    float4 v[NP][kKSplitSlices];
#pragma unroll
    for (int j = 0; j < kKSplitSlices; ++j)
#pragma unroll
        for (int q = 0; q < NP; ++q)
            if (j < run[q].n) v[q][j] = __ldcg(run[q].p + j * kSlotF4);
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int j = 0; j < kKSplitSlices; ++j)
            if (j < run[q].n) {
                s0 += __uint_as_float((uint32_t)bf16_bits(two_float_value(v[q][j].x, v[q][j].y)) << 16);
                s1 += __uint_as_float((uint32_t)bf16_bits(two_float_value(v[q][j].z, v[q][j].w)) << 16);
            }
        y[q] = make_float2(s0, s1);
    }
}

// Small CTAs that fit on an SM next to a stream CTA: with overlap, the finish
// of one step runs under the next step's weight stream, and the next stream
// stores its partials only once this kernel is complete.  Under that load a
// round trip to memory takes microseconds, so a CTA makes as few as it can.
// The grid is at most one CTA per SM: CTA r < rows sums row r's 896 router
// logits (224 threads, two column pairs each) and runs the row's top-16 from
// shared memory; the other CTAs sum latent items (row, 256-column tile) in
// two halves of 128 threads, one column pair per thread, each half taking
// `per_half` (1 or 2) consecutive items per memory round trip.
static_assert(kExpertsTopk == kExperts, "top-16 row width");
constexpr int kRouterThreads = kExperts / 4;    // 224
constexpr int kLatentThreads = kDTileCols / 2;  // 128 per latent item
constexpr int kFinishThreads = 2 * kLatentThreads;

// Latent items per CTA half and round trip: 2 above 16 rows, or when one
// pass over the 14 * rows items at 1 would need more than one CTA per SM;
// else 1.  (Measured: at 20 rows the CTAs that needed two passes made it
// 0.2 us a layer slower; at 17..18 rows 2 is 0.1..0.2 us faster, at 1..16
// rows 1 is as fast or faster.)
int finish_per_half(const DecodeArgs &a) {
    return a.rows > 16 || a.rows + (kDLatTiles * a.rows + 1) / 2 > a.grid ? 2 : 1;
}

// rows router CTAs + enough latent CTAs for one pass over the 14 * rows
// latent items, capped at the stream grid (one CTA per SM), with at least one
// latent CTA.
int finish_grid(const DecodeArgs &a) {
    const int per_cta = 2 * finish_per_half(a);
    int g = a.rows + (kDLatTiles * a.rows + per_cta - 1) / per_cta;
    if (g > a.grid) g = a.grid;
    if (g < a.rows + 1) g = a.rows + 1;
    return g;
}

// The latent CTAs of the finish kernel (KSPLIT: the general path's K-split
// arithmetic).  Pass p: each half sums items i0 .. i0 + per_half - 1, i0 =
// per_half * (2 (p * latent CTAs + CTA) + half), with one memory round trip.
template <bool KSPLIT>
__device__ __forceinline__ void finish_latent(const DecodeArgs &a, int per_half) {
    const int rows = a.rows;
    const int tid = threadIdx.x;
    const int b = blockIdx.x;
    const int n_items = kDLatTiles * rows;
    const int half = tid / kLatentThreads;
    const int cc = 2 * (tid % kLatentThreads);
    const int first = per_half * (2 * (b - rows) + half);
    const int stride = per_half * 2 * ((int)gridDim.x - rows);
    SlotRun run[2];
    auto runs_at = [&](int i0) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int i = i0 + q;
            run[q] = q < per_half && i < n_items ? slot_run(a, i / kDLatTiles, i % kDLatTiles, cc)
                                                 : SlotRun{nullptr, 0};
        }
    };
    runs_at(first);
    pin(run[0]);
    pin(run[1]);
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the stream kernel's partials are complete
    for (int i0 = first; i0 < n_items; i0 += stride) {
        if (i0 != first) runs_at(i0);
        float2 y[2];
        if constexpr (KSPLIT)
            ksplit_slot_pairs<2>(run, y);
        else
            sum_slot_pairs<2, 8>(run, y);  // batches of 8 slots: the registers of two items
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int i = i0 + q;
            if (q >= per_half || i >= n_items) break;  // the same for the whole half
            const int r = i / kDLatTiles, t = i % kDLatTiles;
            const uint16_t b0 = bf16_bits(y[q].x), b1 = bf16_bits(y[q].y);
            if (ROUTE_IN_BOUNDS(r < rows && t < kDLatTiles && cc + 1 < kDTileCols, a.words))
                *reinterpret_cast<uint32_t *>(a.latent + (size_t)r * kLatent + t * kDTileCols + cc) =
                    (uint32_t)b0 | ((uint32_t)b1 << 16);
        }
    }
}

// The router CTA of row r: sums the row's 896 router logits (224 threads,
// two column pairs each), stores them and, with do_topk, runs the row's
// top-16 (a3/a4) with all 224 threads.  Threads 224.. do not call it.
__device__ __forceinline__ void finish_router(const DecodeArgs &a, int r, int do_topk,
                                              TopkBlockSmem &s_topk) {
    const int tid = threadIdx.x;
    const int c0 = 2 * tid, c1 = c0 + kExperts / 2;  // columns c0, c0+1 and c1, c1+1
    SlotRun run[2] = {slot_run(a, r, kDLatTiles + c0 / kDTileCols, c0 % kDTileCols),
                      slot_run(a, r, kDLatTiles + c1 / kDTileCols, c1 % kDTileCols)};
    pin(run[0]);
    pin(run[1]);
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the stream kernel's partials are complete
    float2 y[2];
    sum_slot_pairs<2>(run, y);
    float *lrow = a.logits + (size_t)r * kExperts;
    if (!ROUTE_IN_BOUNDS(r < a.rows && c1 + 1 < kExperts, a.words)) return;
    *reinterpret_cast<float2 *>(lrow + c0) = y[0];
    *reinterpret_cast<float2 *>(lrow + c1) = y[1];
    if (!do_topk) return;
    // the heavy-tie fallback re-reads the logits this CTA just stored,
    // ordered by the top-16's barriers
    const float v[4] = {y[0].x, y[0].y, y[1].x, y[1].y};
    const int id[4] = {c0, c0 + 1, c1, c1 + 1};
    topk16_block(v, id, lrow, tid, 1, s_topk, a.ids + (size_t)r * kTopK,
                 a.weights + (size_t)r * kTopK);
}

__global__ void __maxnreg__(112) decode_finish_kernel(const __grid_constant__ DecodeArgs a,
                                                      int do_topk, int per_half) {
    __shared__ TopkBlockSmem s_topk;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int b = blockIdx.x;
    if (b < a.rows) {
        if (threadIdx.x < kRouterThreads) finish_router(a, b, do_topk, s_topk);
    } else if (a.ksplit) {
        finish_latent<true>(a, per_half);
    } else {
        finish_latent<false>(a, per_half);
    }
}

// The finish kernel when the latent sum of squares is asked for ("Optionally
// gather the Kimi3 prefill latent instead of reducing it", Reviewer Notes:
// the FP32 statistic the latent norm needs), as one thread-block cluster per
// row: rank 0 is the row's router CTA, ranks 1.. its latent CTAs, each
// taking 2 per_half consecutive tiles of the row (two halves of 128 threads,
// per_half tiles each, one memory round trip).  Every latent item adds the
// squares of the 256 BF16 values it stores (exact in FP32) as a two-float in
// a fixed order (warp tree, then its 4 warps in order) and writes that part
// into rank 0's shared memory; each latent CTA then arrives once on rank 0's
// barrier and leaves.  Rank 0, after its top-16, waits for every arrival,
// adds the row's 14 parts in tile order and rounds once.  No global counter
// and no second pass over memory: the parts meet in distributed shared
// memory while the router CTA runs the top-16 (measured: +0.14 us a layer at
// 8 rows, +0.21 us at 20 rows, against +0.87 / +2.10 us for parts summed
// through a per-row arrival counter in global memory, and +1.38 / +1.46 us
// when the latent CTAs stayed until a final cluster barrier).  Rank 0 can
// only stop waiting after a bound four times the kernels' own: the latent
// CTAs have no wait but the grid dependency, which ends with the stream
// kernel and its bounded waits.
__host__ __device__ constexpr int ss_latent_ctas(int per_half) {
    return (kDLatTiles + 2 * per_half - 1) / (2 * per_half);
}

template <bool KSPLIT>
__global__ void __maxnreg__(112) decode_finish_ss_kernel(const __grid_constant__ DecodeArgs a,
                                                         int do_topk, int per_half) {
    __shared__ TopkBlockSmem s_topk;
    __shared__ float2 s_ss[2][2][kLatentThreads / 32];  // [item][half][warp]
    __shared__ float2 s_part[kDLatTiles];               // rank 0: the row's parts, by tile
    __shared__ __align__(8) uint64_t s_bar;             // rank 0: one arrival per latent CTA
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x;
    const uint32_t rank = ptx::cluster_ctarank();
    const int nlat = ss_latent_ctas(per_half);
    const int r = blockIdx.x / (1 + nlat);
    const uint32_t bar = ptx::smem_addr(&s_bar);
    if (rank == 0 && tid == 0) {
        ptx::mbar_init(bar, (uint32_t)nlat);
        ptx::fence_barrier_init();
    }
    ptx::cluster_sync();  // every CTA of the cluster runs and rank 0's barrier is initialised
    if (rank == 0) {
        if (tid < kRouterThreads) finish_router(a, r, do_topk, s_topk);
    } else {
        const int half = tid / kLatentThreads, ht = tid % kLatentThreads, cc = 2 * ht;
        const int t0 = ((int)rank - 1) * 2 * per_half + half * per_half;
        SlotRun run[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int t = t0 + q;
            run[q] = q < per_half && t < kDLatTiles ? slot_run(a, r, t, cc) : SlotRun{nullptr, 0};
        }
        pin(run[0]);
        pin(run[1]);
        asm volatile("griddepcontrol.wait;" ::: "memory");  // the stream kernel's partials are complete
        float2 y[2];
        if constexpr (KSPLIT)
            ksplit_slot_pairs<2>(run, y);
        else
            sum_slot_pairs<2, 8>(run, y);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int t = t0 + q;
            if (q >= per_half || t >= kDLatTiles) break;  // the same for the whole half
            const uint16_t b0 = bf16_bits(y[q].x), b1 = bf16_bits(y[q].y);
            if (ROUTE_IN_BOUNDS(r < a.rows && cc + 1 < kDTileCols, a.words))
                *reinterpret_cast<uint32_t *>(a.latent + (size_t)r * kLatent + t * kDTileCols + cc) =
                    (uint32_t)b0 | ((uint32_t)b1 << 16);
            const float v0 = __uint_as_float((uint32_t)b0 << 16);
            const float v1 = __uint_as_float((uint32_t)b1 << 16);
            float hi = v0 * v0, lo = 0.f;
            two_sum_acc(hi, lo, v1 * v1);
            warp_two_sum(hi, lo);
            if ((ht & 31) == 0) s_ss[q][half][ht >> 5] = make_float2(hi, lo);
        }
        if (half == 0)
            asm volatile("barrier.sync 2, %0;" ::"n"(kLatentThreads) : "memory");
        else
            asm volatile("barrier.sync 3, %0;" ::"n"(kLatentThreads) : "memory");
        if (ht == 0) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int t = t0 + q;
                if (q >= per_half || t >= kDLatTiles) break;
                float hi = s_ss[q][half][0].x, lo = s_ss[q][half][0].y;
#pragma unroll
                for (int w = 1; w < kLatentThreads / 32; ++w) {
                    two_sum_acc(hi, lo, s_ss[q][half][w].x);
                    lo += s_ss[q][half][w].y;
                }
                ptx::st_cluster_f2(ptx::map_to_rank(ptx::smem_addr(&s_part[t]), 0u),
                                   make_float2(hi, lo));
            }
        }
        __syncthreads();  // both halves' parts written
        if (tid == 0) ptx::mbar_arrive_remote(ptx::map_to_rank(bar, 0u));
        return;
    }
    if (tid != 0) return;
    // rank 0 waits for every latent CTA's arrival (after its own top-16)
    const uint64_t t0 = ptx::global_timer_ns();
    bool ok = true;
    while (!ptx::mbar_try_wait_cluster(bar, 0u)) {
        if (ptx::global_timer_ns() - t0 > 4 * a.timeout_ns) {
            atomicOr(a.words, kStatusTimeout);
            ok = false;
            break;
        }
    }
    if (ok && ROUTE_IN_BOUNDS(r < a.rows, a.words)) {
        float hi = s_part[0].x, lo = s_part[0].y;
#pragma unroll
        for (int t = 1; t < kDLatTiles; ++t) {
            two_sum_acc(hi, lo, s_part[t].x);
            lo += s_part[t].y;
        }
        a.sumsq[r] = two_float_value(hi, lo);
    }
}

// The finish of a column shard at decode sizes.  A shard's few column tiles
// are streamed by many CTAs, so a value may have up to 64 partials: each
// column pair is summed by S = 1, 2 or 4 neighbouring threads (`split`),
// thread j of the S taking the j-th run of at most 16 consecutive slots (one
// memory round trip), and the S two-floats are joined by a fixed shuffle
// tree (j = 0 with 1 and 2 with 3, then the two), so that every value's bits
// depend on the plan only.  CTA r < rows sums row r's n_exp router logits,
// stores them, and its first warp picks the shard's top-16 of them as
// candidates (the same selection as the standalone shard top-16); the other
// CTAs take (row, latent tile, quarter of the tile's column pairs per
// `split`) items and store the latent columns below n_lat.
struct PairSum {
    float2 hi, lo;  // the pair's two columns
};

__device__ __forceinline__ PairSum sum_slot_range(const float4 *p, int n) {
    PairSum r{make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    float4 v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
        if (j < n) v[j] = __ldcg(p + j * kSlotF4);
#pragma unroll
    for (int j = 0; j < 16; ++j)
        if (j < n) {
            two_sum_acc(r.hi.x, r.lo.x, v[j].x);
            r.lo.x += v[j].y;
            two_sum_acc(r.hi.y, r.lo.y, v[j].z);
            r.lo.y += v[j].w;
        }
    return r;
}

// Joins the two-floats of the `split` threads of a pair (lanes aligned to
// `split`); the pair's first thread ends with the total.
__device__ __forceinline__ void join_split(PairSum &s, int split) {
    for (int off = 1; off < split; off <<= 1) {
        const float hx = __shfl_down_sync(0xFFFFFFFFu, s.hi.x, off);
        const float hy = __shfl_down_sync(0xFFFFFFFFu, s.hi.y, off);
        const float lx = __shfl_down_sync(0xFFFFFFFFu, s.lo.x, off);
        const float ly = __shfl_down_sync(0xFFFFFFFFu, s.lo.y, off);
        two_sum_acc(s.hi.x, s.lo.x, hx);
        s.lo.x += lx;
        two_sum_acc(s.hi.y, s.lo.y, hy);
        s.lo.y += ly;
    }
}

// Thread j of the `split` threads of column pair cc of tile t, row r: its
// run of the tile's slots.
__device__ __forceinline__ SlotRun split_run(const DecodeArgs &a, int r, int t, int cc, int split,
                                             int j) {
    SlotRun run = slot_run(a, r, t, cc);
    const int per = (run.n + split - 1) / split;
    const int s0 = j * per < run.n ? j * per : run.n;
    const int s1 = s0 + per < run.n ? s0 + per : run.n;
    run.p += (size_t)s0 * kSlotF4;
    run.n = s1 - s0;
    return run;
}

__global__ void __maxnreg__(112)
    decode_shard_finish_kernel(const __grid_constant__ DecodeArgs a, int n_lat, int n_exp,
                               int id_base, int32_t *__restrict__ cand_ids,
                               float *__restrict__ cand_logits, int split) {
    __shared__ uint2 s_cand[kCandMax];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x;
    const int b = blockIdx.x;
    const int rows = a.rows;
    const int j = tid % split;
    if (b < rows) {
        const int r = b;
        float *lrow = a.logits + (size_t)r * n_exp;
        asm volatile("griddepcontrol.wait;" ::: "memory");  // the stream kernel's partials are complete
        const int pairs = n_exp / 2;
        for (int i0 = 0; i0 < pairs * split; i0 += kFinishThreads) {  // whole warps in every pass
            const int i = i0 + tid, c = 2 * (i / split);
            const bool mine = c < n_exp;
            SlotRun run = mine ? split_run(a, r, a.lat_tiles + c / kDTileCols, c % kDTileCols, split, j)
                               : SlotRun{nullptr, 0};
            PairSum ps = sum_slot_range(run.p, run.n);
            join_split(ps, split);
            if (mine && j == 0 && ROUTE_IN_BOUNDS(c + 1 < n_exp, a.words))
                *reinterpret_cast<float2 *>(lrow + c) = make_float2(
                    two_float_value(ps.hi.x, ps.lo.x), two_float_value(ps.hi.y, ps.lo.y));
        }
        __syncthreads();  // the row's logits are stored
        if (tid < 32) {
            uint32_t key, id;
            topk16_warp_picks(lrow, n_exp, tid, s_cand, key, id);
            if (tid < kTopK) {
                cand_ids[(size_t)r * kTopK + tid] = id_base + (int32_t)id;
                cand_logits[(size_t)r * kTopK + tid] = key_to_float(key);
            }
        }
    } else {
        // item (row, tile, part): part q covers column pairs q * 256 / split ..
        const int parts = split > 2 ? split / 2 : 1;
        const int i = b - rows, q = i % parts, t = (i / parts) % a.lat_tiles,
                  r = i / (parts * a.lat_tiles);
        const int cc = 2 * (q * (kFinishThreads / split) + tid / split), col = t * kDTileCols + cc;
        const bool mine = cc < kDTileCols && col < n_lat;
        SlotRun run = mine ? split_run(a, r, t, cc, split, j) : SlotRun{nullptr, 0};
        pin(run);
        asm volatile("griddepcontrol.wait;" ::: "memory");  // the stream kernel's partials are complete
        PairSum ps = sum_slot_range(run.p, run.n);
        join_split(ps, split);
        if (mine && j == 0 && ROUTE_IN_BOUNDS(r < rows && col + 1 < n_lat, a.words))
            *reinterpret_cast<uint32_t *>(a.latent + (size_t)r * n_lat + col) =
                (uint32_t)bf16_bits(two_float_value(ps.hi.x, ps.lo.x)) |
                ((uint32_t)bf16_bits(two_float_value(ps.hi.y, ps.lo.y)) << 16);
    }
}

cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t c = {};
    c.gridDim = grid;
    c.blockDim = block;
    c.dynamicSmemBytes = smem;
    c.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    c.attrs = attr;
    c.numAttrs = 1;
    return c;
}

template <int BN>
cudaError_t configure_bn() {
    return cudaFuncSetAttribute(decode_stream_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)DecCfg<BN>::kSmemBytes);
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap &mh, const CUtensorMap &ml, const CUtensorMap &mr,
                      const DecodeArgs &a, cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t c =
        pdl_config(dim3(a.grid), dim3(kDecThreads), DecCfg<BN>::kSmemBytes, stream, attr);
    return cudaLaunchKernelEx(&c, decode_stream_kernel<BN>, mh, ml, mr, a);
}

}  // namespace

int decode_bn_for(int rows) { return rows <= 16 ? 16 : 32; }

int decode_smem_bytes(int bn) {
    return bn == 16 ? (int)DecCfg<16>::kSmemBytes : bn == 32 ? (int)DecCfg<32>::kSmemBytes : -1;
}

cudaError_t decode_configure(int bn) {
    return bn == 16 ? configure_bn<16>() : bn == 32 ? configure_bn<32>() : cudaErrorInvalidValue;
}

cudaError_t decode_shard_launch(int bn, const CUtensorMap &map_h, const CUtensorMap &map_wl,
                                const CUtensorMap &map_wr, const DecodeArgs &args, int n_lat,
                                int n_exp, int id_base, int32_t *cand_ids, float *cand_logits,
                                cudaStream_t stream) {
    if (n_exp < kTopK || n_exp > kExpertsTopk || args.lat_tiles < 1) return cudaErrorInvalidValue;
    int most = 0;  // partials of a value: the CTAs covering a tile
    for (int t = 0; t < args.tiles; ++t) most = args.seg_count[t] > most ? args.seg_count[t] : most;
    const int split = most <= 16 ? 1 : most <= 32 ? 2 : most <= 64 ? 4 : 0;
    if (split == 0) return cudaErrorInvalidValue;
    cudaError_t e = bn == 16   ? launch_bn<16>(map_h, map_wl, map_wr, args, stream)
                    : bn == 32 ? launch_bn<32>(map_h, map_wl, map_wr, args, stream)
                               : cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    const int parts = split > 2 ? split / 2 : 1;  // CTAs per (row, latent tile)
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t c = pdl_config(dim3(args.rows * (1 + args.lat_tiles * parts)),
                                      dim3(kFinishThreads), 0, stream, attr);
    return cudaLaunchKernelEx(&c, decode_shard_finish_kernel, args, n_lat, n_exp, id_base, cand_ids,
                              cand_logits, split);
}

cudaError_t decode_launch(int bn, const CUtensorMap &map_h, const CUtensorMap &map_wl,
                          const CUtensorMap &map_wr, const DecodeArgs &args, int do_topk,
                          cudaStream_t stream) {
    cudaError_t e = bn == 16   ? launch_bn<16>(map_h, map_wl, map_wr, args, stream)
                    : bn == 32 ? launch_bn<32>(map_h, map_wl, map_wr, args, stream)
                               : cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    const int per_half = finish_per_half(args);
    if (args.sumsq == nullptr) {
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t c =
            pdl_config(dim3(finish_grid(args)), dim3(kFinishThreads), 0, stream, attr);
        return cudaLaunchKernelEx(&c, decode_finish_kernel, args, do_topk, per_half);
    }
    // one cluster per row: the router CTA and its latent CTAs
    const int csize = 1 + ss_latent_ctas(per_half);
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t c =
        pdl_config(dim3(args.rows * csize), dim3(kFinishThreads), 0, stream, attr);
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)csize;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    c.numAttrs = 2;
    return args.ksplit ? cudaLaunchKernelEx(&c, decode_finish_ss_kernel<true>, args, do_topk, per_half)
                       : cudaLaunchKernelEx(&c, decode_finish_ss_kernel<false>, args, do_topk, per_half);
}

}  // namespace route
