// Prefill route projection (steps a1 and a2 for a chunk of token rows) on
// the sm_103a tensor cores, two SMs per tile.
//
//   latent[r, n] = bf16( sum_k hidden[r, k] * W_latent[k, n] )   n < 3584
//   logits[r, e] =       sum_k hidden[r, k] * W_router[k, e]    e < 896
//
// Each latent value is one FP32-accumulated dot product over the full K =
// 7168, rounded once ("Optionally gather the Kimi3 prefill latent instead of
// reducing it", Description, Numerics and Compile bullets: at prefill the
// projection is a dense M = rows, K = 7168 GEMM); the two projections share
// the hidden operand and run as one N = 3584 + 896 problem.
//
// The weights are [K, N] with N contiguous, so their tensor-core operand is
// MN-major.  A tile is 256 weight columns (the MMA's M) by 256 token rows
// (its N), computed by a cluster of two CTAs with
// tcgen05.mma.cta_group::2: each CTA stages its 128 weight columns (A) and
// its half of the token rows (B) per 64-deep k-block, and holds its 128
// weight columns x N token rows of the FP32 accumulator in its own TMEM.
//
// Tile kinds (the host builds each pair's list; see common.cuh):
//   plain: one accumulation over the whole K; the epilogue stores the latent
//     (rounded to BF16, with per-row sum-of-squares parts when asked) or the
//     FP32 router logits.  Columns past the plan's latent or expert count (a
//     column shard's share, or 896 experts in four 256-column tiles) are not
//     stored.
//   K-split (latent): the general path's eight 896-deep K slices (same page,
//     Numerics bullet and commit body) as eight jobs, each slice's result
//     rounded to BF16 and added in FP32, in slice order, to a running sum the
//     epilogue keeps in registers (128 a thread).
// Every job accumulates 256 TMEM columns, an aligned pair of quarters, and
// the pairs {0,1} and {2,3} alternate from job to job, so one job is drained
// while the next is computed.
//
// Warp roles (320 threads, persistent, one CTA per SM, pairs = clusters):
//   warp 0      TMA producer (both CTAs); completion is counted on the leader
//               CTA's barrier, which the leader arms for both CTAs' bytes
//               before either may fill the stage
//   warp 1      TMEM owner (both CTAs); the leader's lane 0 issues the MMAs
//               and re-arms each stage's barrier once it has consumed it
//   warps 2..9  epilogue (both CTAs): warp w reads TMEM lanes 32 (w % 4) ..
//               +31 and half of the tile's token rows; results go through a
//               small shared-memory buffer per warp and out with TMA stores
//               (32 columns x 16 rows per store).
//
// Programmatic dependent launch: weight boxes of the first stages are
// requested before `griddepcontrol.wait` (no predecessor writes the weights);
// outputs are written only after it, and hidden rows are read only after it
// too unless `overlap` is set.
//
// Every wait is bounded: after args.timeout_ns a waiting thread sets the
// device status word and the CTA's abort flag, in-flight copies and MMAs are
// drained, TMEM is freed and the CTA returns (both CTAs of a pair meet at a
// final cluster barrier, so neither leaves while the other may still reach
// its shared memory).
#include <cuda_bf16.h>
#include <type_traits>

#include "common.cuh"
#include "sm103_ptx.cuh"
#include "twofloat.cuh"

namespace route {
namespace {

constexpr uint32_t kBoxBytes = 64 * 64 * 2;                // 64 x 64 BF16 box
constexpr int kHalf = 128;                                 // each CTA's weight columns
constexpr uint32_t kBBytes = 2 * kBoxBytes;                // up to 128 token rows x 64 k
constexpr uint32_t kABytes = 2 * kBoxBytes;                // 128 weight columns x 64 k
constexpr uint32_t kStageBytes = kBBytes + kABytes;        // B first, then A
constexpr int kStages = 6;
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr uint32_t kStoreBufBytes = 16 * 32 * 4;           // 16 rows x 32 columns, up to FP32
constexpr uint32_t kStoreBytes = kEpiWarps * 2 * kStoreBufBytes;
constexpr uint32_t kSmemBytes = 1024 + kStages * kStageBytes + kStoreBytes + 256;
constexpr uint32_t kTmemCols = 512;                        // four quarters of 128 columns
static_assert(kMaxPairTiles >= 64, "tile list");

// tcgen05 instruction descriptor, kind::f16: FP32 accumulator, BF16 A and B,
// A MN-major (transposed), B K-major, M = 256 (over the pair), N = n.
constexpr uint32_t idesc_for(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(2 * kHalf >> 4) << 24);
}
constexpr uint32_t kIdesc = idesc_for(kPrefillBN);
static_assert(kProjThreads == 64 + kEpiThreads, "warp roles");
static_assert(kHalf == 2 * kPrefillHiddenBoxRows, "two hidden boxes per CTA and full tile");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
static_assert(8 * (2 * kStages + 9) <= 256, "barrier area");
static_assert(kLatent == kPrefillLatTiles * 2 * kHalf, "latent tiles");

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile.
// lbo / sbo are the leading / stride byte offsets of the canonical layout.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;  // descriptor version for tcgen05
    d |= 2ull << 61;  // 128-byte swizzle
    return d;
}

__device__ __forceinline__ int tile_jobs(int kind) { return kind == kTileFull ? 1 : kKSplitSlices; }

// Transaction bytes of one stage, both CTAs.
constexpr uint32_t kStageTx = 2u * kStageBytes;

// Bounded wait for the completion of phase `parity` of `bar` (acquire at
// cluster scope: other CTAs of the pair arrive on these barriers).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const ProjArgs &a,
                                           volatile int *abort_flag) {
    if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = ptx::global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 63u) == 0u) {
            if (*abort_flag) return false;
            if (ptx::global_timer_ns() - t0 > a.timeout_ns) {
                *abort_flag = 1;
                atomicOr(a.status, kStatusTimeout);
                return false;
            }
        }
    }
}

// Bounded wait used only while tearing down.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, const ProjArgs &a) {
    const uint64_t t0 = ptx::global_timer_ns();
    while (!ptx::mbar_try_wait_cluster(bar, parity)) {
        if (ptx::global_timer_ns() - t0 > a.timeout_ns) {
            atomicOr(a.status, kStatusTimeout);
            return;
        }
    }
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ float bf16_round(float x) {
    return __uint_as_float((uint32_t)bf16_bits(x) << 16);
}

// 168 registers a thread (320 threads, one CTA an SM): with this cap as
// __maxnreg__ nothing spills, where __launch_bounds__(320, 1) spilled a few
// words in the K-split epilogue
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(168)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap map_h,
                        const __grid_constant__ CUtensorMap map_wl,
                        const __grid_constant__ CUtensorMap map_wr,
                        const __grid_constant__ CUtensorMap map_lat,
                        const __grid_constant__ CUtensorMap map_lg,
                        const __grid_constant__ ProjArgs args) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem_base;
    __shared__ volatile int s_abort;
    __shared__ int s_tiles[kMaxPairTiles];  // this pair's tile list (read every k-block)

    // Both CTAs of a pair lay out shared memory identically, so an offset in
    // one names the same operand or barrier in the other.
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    const uint32_t store_base = sbase + kStages * kStageBytes;
    const uint32_t bars = store_base + kStoreBytes;
    auto full_bar = [&](int s) { return bars + 8u * s; };                 // leader's are used
    auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
    auto qfull_bar = [&](int q) { return bars + 8u * (2 * kStages + q); };
    auto qempty_bar = [&](int q) { return bars + 8u * (2 * kStages + 4 + q); };  // leader's
    const uint32_t drain_bar = bars + 8u * (2 * kStages + 8);

    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = rank == 0u;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int pair = blockIdx.x >> 1;
    const int tile0 = args.sched_off[pair];
    const int ntiles = args.sched_off[pair + 1] - tile0;
    const int total = ntiles * kKBlocks;
    const int *const sched = s_tiles;
    for (int i = threadIdx.x; i < ntiles; i += blockDim.x)
        if (ROUTE_IN_BOUNDS(i < kMaxPairTiles, args.status)) s_tiles[i] = args.sched[tile0 + i];
    __syncthreads();

    if (threadIdx.x == 0) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        s_abort = 0;
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int q = 0; q < 4; ++q) {
            ptx::mbar_init(qfull_bar(q), 1);
            ptx::mbar_init(qempty_bar(q), 2 * kEpiWarps);  // each epilogue warp of both CTAs
        }
        ptx::mbar_init(drain_bar, 1);
        // the leader arms the first round of every stage that will be filled
        // (all of them belong to the pair's first tile)
        const int first = total < kStages ? total : kStages;
        if (leader && ntiles > 0)
            for (int s = 0; s < first; ++s)
                ptx::mbar_arrive_expect_tx(full_bar(s), kStageTx);
        ptx::fence_barrier_init();
        ptx::prefetch_tensormap(&map_h);
        ptx::prefetch_tensormap(&map_wl);
        ptx::prefetch_tensormap(&map_wr);
        ptx::prefetch_tensormap(&map_lat);
        ptx::prefetch_tensormap(&map_lg);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_addr(&s_tmem_base), kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
    ptx::tc_fence_after();
    const uint32_t tmem_base = s_tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            // The pairs at work share a band's weight tiles while the hidden
            // rows are read again by every band: weights go first when L2
            // needs room (measured at 3072 rows: 156 MB of DRAM reads a
            // launch against 207 MB with the default policy, 3% faster
            // under the power cap).
            const uint64_t pol_w = ptx::policy_evict_first();
            const uint64_t pol_h = ptx::policy_evict_last();
            uint32_t armed = 0u, armed_par = 0u;  // leader: stages armed / their phase parity
            const int n_pre = total < kStages ? total : kStages;
            auto weights_of = [&](int it, uint32_t st, uint32_t bar) {
                const int t = sched[it / kKBlocks];
                const int kb = it % kKBlocks;
                const int c = tile_col(t);
                const bool lat = c < kPrefillLatTiles;
                const CUtensorMap *wmap = lat ? &map_wl : &map_wr;
                // this CTA's 128 columns; past column 896 of W_router TMA fills zeros
                const int x0 = (lat ? c : c - kPrefillLatTiles) * 2 * kHalf + (int)rank * kHalf;
                ptx::tma_load_2d_pair(st + kBBytes, wmap, bar, x0, kb * kKBlock, pol_w);
                ptx::tma_load_2d_pair(st + kBBytes + kBoxBytes, wmap, bar, x0 + 64, kb * kKBlock,
                                      pol_w);
            };
            auto hidden_of = [&](int it, uint32_t st, uint32_t bar) {  // this CTA's 128 of 256 rows
                const int y0 = tile_row0(sched[it / kKBlocks]) + (int)rank * kHalf;
                const int k0 = (it % kKBlocks) * kKBlock;
                ptx::tma_load_2d_pair(st, &map_h, bar, k0, y0, pol_h);
                ptx::tma_load_2d_pair(st + kBoxBytes, &map_h, bar, k0, y0 + 64, pol_h);
            };
            // Weight boxes of the first stages go out before the grid
            // dependency resolves (no predecessor writes the weights).
            for (int it = 0; it < n_pre; ++it) {
                weights_of(it, sbase + it * kStageBytes, ptx::map_to_rank(full_bar(it), 0u));
                armed |= 1u << it;
            }
            if (!args.overlap) asm volatile("griddepcontrol.wait;" ::: "memory");
            for (int it = 0; it < n_pre; ++it) {
                if (args.test_stall && leader && it == total - 1) continue;  // test hook
                hidden_of(it, sbase + it * kStageBytes, ptx::map_to_rank(full_bar(it), 0u));
            }
            bool ok = true;
            for (int it = n_pre; it < total; ++it) {
                const int s = it % kStages;
                const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                if (!wait_phase(empty_bar(s), ph ^ 1u, args, &s_abort)) {
                    ok = false;
                    break;
                }
                if (args.test_stall && leader && it == total - 1) continue;  // test hook
                const uint32_t st = sbase + s * kStageBytes;
                const uint32_t fb = ptx::map_to_rank(full_bar(s), 0u);
                weights_of(it, st, fb);
                hidden_of(it, st, fb);
                armed |= 1u << s;
                armed_par = (armed_par & ~(1u << s)) | (ph << s);
            }
            // After an abort the leader lets every copy it armed land (the
            // peer's copies complete on the same barriers).
            if (leader && (!ok || s_abort)) {
                for (int s = 0; s < kStages; ++s)
                    if (armed & (1u << s)) wait_drain(full_bar(s), (armed_par >> s) & 1u, args);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (leader CTA) ----------------
            uint32_t occ = 0u;  // bit q: parity of the occupations of TMEM quarter q so far
            auto acquire = [&](int q) {
                const bool r = wait_phase(qempty_bar(q), ((occ >> q) & 1u) ^ 1u, args, &s_abort);
                occ ^= 1u << q;
                return r;
            };
            int it = 0, job = 0;
            bool ok = true;
            for (int i = 0; i < ntiles && ok; ++i) {
                const int njobs = tile_jobs(tile_kind(sched[i]));
                const int kbpj = kKBlocks / njobs;  // k-blocks of one job
                for (int j = 0; j < njobs && ok; ++j, ++job) {
                    const int q = 2 * (job & 1);
                    if (!(acquire(q) && acquire(q + 1))) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (uint32_t)(128 * q);
                    for (int kb = 0; kb < kbpj; ++kb, ++it) {
                        const int s = it % kStages;
                        const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                        if (!wait_phase(full_bar(s), ph, args, &s_abort)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t b = sbase + s * kStageBytes;
                        const uint32_t a = b + kBBytes;
#pragma unroll
                        for (int kk = 0; kk < kKBlock / 16; ++kk) {
                            // A: k advances 16 rows = two 8-row swizzle atoms (2048 B);
                            //    the two 64-column boxes are 8192 B apart (LBO),
                            //    8-row k groups 1024 B apart (SBO).
                            // B: k advances 32 B inside the 128-byte swizzled row;
                            //    8-row groups of token rows are 1024 B apart (SBO).
                            const uint64_t da = smem_desc(a + kk * 2048u, kBoxBytes, 1024u);
                            const uint64_t db = smem_desc(b + kk * 32u, 16u, 1024u);
                            ptx::mma_bf16_pair(d_tmem, da, db, kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
                        }
                        // re-arm stage s for its next round before it is freed:
                        // the copies that fill it can only start after the commit
                        if (it + kStages < total) ptx::mbar_arrive_expect_tx(full_bar(s), kStageTx);
                        ptx::mma_commit_pair(empty_bar(s), 0x3);  // frees stage s in both CTAs
                    }
                    if (ok) ptx::mma_commit_pair(qfull_bar(q), 0x3);
                }
            }
            ptx::mma_commit_pair(drain_bar, 0x3);  // every MMA retired before TMEM is freed
            wait_drain(drain_bar, 0u, args);
        }
    } else {
        // ---------------- epilogue (warps 2..9, both CTAs) ----------------
        const int lq = warp & 3;            // TMEM lanes 32*lq .. +31 = this CTA's weight columns
        const int cs = (warp - 2) >> 2;     // which half of the tile's token rows
        const int rows = args.rows;
        const uint32_t lanes = tmem_base + ((uint32_t)(32 * lq) << 16);
        uint8_t *const store_gen = smem_raw + (store_base - raw) + (warp - 2) * 2 * kStoreBufBytes;
        const uint32_t store_sh = store_base + (warp - 2) * 2 * kStoreBufBytes;
        int sb = 0;
        uint32_t qc = 0u;  // bit q: parity of the completions of quarter q consumed
        int job = 0;       // jobs so far: job j accumulates in quarters 2 (j & 1) and 2 (j & 1) + 1
        asm volatile("griddepcontrol.wait;" ::: "memory");  // outputs may still be read by the predecessor

        // Stage 16 rows of this warp's 32 columns and send them out with one
        // TMA store (rows past `rows` and columns past the map are not written).
        auto store_chunk = [&](const uint32_t (&v)[16], bool fp32, const CUtensorMap *map, int x,
                               int y, bool valid) {
            if (lane == 0) ptx::bulk_wait_group_read<1>();  // this buffer's last store has read it
            __syncwarp();
            uint8_t *buf = store_gen + sb * kStoreBufBytes;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                if (fp32)
                    reinterpret_cast<uint32_t *>(buf)[jj * 32 + lane] = v[jj];
                else
                    reinterpret_cast<uint16_t *>(buf)[jj * 32 + lane] = (uint16_t)v[jj];
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (valid && y < rows && ROUTE_IN_BOUNDS(y >= 0 && (x & 31) == 0, args.status))
                    ptx::tma_store_2d(map, store_sh + sb * kStoreBufBytes, x, y);
                // one group per chunk, empty when nothing is stored, so that
                // "at most one group pending" always means this buffer is free
                ptx::bulk_commit_group();
            }
            sb ^= 1;
        };
        // Per-row sum of squares of the 32 BF16 values this warp just staged
        // for rows y .. y + 15 (exact squares; lanes 2r and 2r + 1 take 16
        // values of row r each, joined in a fixed order): one part per row.
        // Packed: even and odd columns as two two-float streams in FP32
        // pairs (half the instructions); the K-split tiles, whose 128 sums
        // are still live here, take the scalar form, which needs fewer
        // registers.  Reads the staging buffer before it can be written again.
        auto sumsq_parts = [&](int part, int y, auto packed) {
            const uint4 *row = reinterpret_cast<const uint4 *>(
                store_gen + (sb ^ 1) * kStoreBufBytes + (lane >> 1) * 64 + (lane & 1) * 32);
            float hi = 0.f, lo = 0.f;
            if constexpr (decltype(packed)::value) {
                uint64_t hi2 = 0u, lo2 = 0u;  // +0.0f in both halves
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    const uint4 w4 = row[g];
                    const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint64_t x = ptx::f32x2_pack(__uint_as_float(w[e] << 16),
                                                           __uint_as_float(w[e] & 0xFFFF0000u));
                        two_sum_acc_x2(hi2, lo2, ptx::f32x2_mul(x, x));
                    }
                }
                float hb, lb;
                ptx::f32x2_unpack(hi2, hi, hb);
                ptx::f32x2_unpack(lo2, lo, lb);
                two_sum_acc(hi, lo, hb);
                lo += lb;
            } else {
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    const uint4 w4 = row[g];
                    const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float a = __uint_as_float(w[e] << 16),
                                    b = __uint_as_float(w[e] & 0xFFFF0000u);
                        two_sum_acc(hi, lo, a * a);
                        two_sum_acc(hi, lo, b * b);
                    }
                }
            }
            const float ohi = __shfl_xor_sync(0xFFFFFFFFu, hi, 1);
            const float olo = __shfl_xor_sync(0xFFFFFFFFu, lo, 1);
            if ((lane & 1) == 0) {
                two_sum_acc(hi, lo, ohi);
                lo += olo;
                if (y + (lane >> 1) < rows &&
                    ROUTE_IN_BOUNDS(y >= 0 && part >= 0 && part < kSsParts, args.status))
                    args.ss_part[(size_t)(y + (lane >> 1)) * kSsParts + part] = make_float2(hi, lo);
            }
        };
        // This warp is done reading quarter q (one of the 16 arrivals the
        // leader's barrier counts: every epilogue warp of both CTAs).
        auto release = [&](int q) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    ptx::mbar_arrive(qempty_bar(q));
                else
                    ptx::mbar_arrive_remote(ptx::map_to_rank(qempty_bar(q), 0u));
            }
        };
        auto wait_full = [&](int q) {
            const bool ok = wait_phase(qfull_bar(q), (qc >> q) & 1u, args, &s_abort);
            qc ^= 1u << q;
            __syncwarp();  // the TMEM loads that follow are warp-wide (.sync.aligned)
            ptx::tc_fence_after();
            return ok;
        };
        bool go = true;
        for (int i = 0; i < ntiles && go; ++i) {
            const int t = sched[i];
            const int c = tile_col(t), kind = tile_kind(t), row0 = tile_row0(t);
            const bool lat = c < kPrefillLatTiles;
            // global column of lane 0 of this warp
            const int xw = (lat ? c : c - kPrefillLatTiles) * 2 * kHalf + (int)rank * kHalf + 32 * lq;
            const bool valid = xw < (lat ? args.n_latent : args.n_experts);
            const int part = c * 8 + (int)rank * 4 + lq;
            const uint32_t acc0 = lanes + (uint32_t)(128 * cs);  // this warp's token rows 128 cs ..
            if (kind == kTileFull) {
                const int q = 2 * (job++ & 1);
                if (!wait_full(q)) {
                    go = false;
                    break;
                }
#pragma unroll 1
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t u[16];
                    ptx::tmem_ld_x16(acc0 + (uint32_t)(128 * q + 16 * ch), u);
                    ptx::tmem_ld_wait();
                    if (ch == 7) {  // every column of the accumulator is in registers
                        release(q);
                        release(q + 1);
                    }
                    const int y = row0 + 128 * cs + 16 * ch;
                    if (lat) {
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) u[jj] = bf16_bits(__uint_as_float(u[jj]));
                        store_chunk(u, false, &map_lat, xw, y, valid);
                        if (args.ss_part != nullptr) sumsq_parts(part, y, std::true_type{});
                    } else {
                        store_chunk(u, true, &map_lg, xw, y, valid);
                    }
                }
            } else {
                // K-split latent: the BF16-rounded slice partials of this
                // warp's 128 token rows, added in FP32 in slice order.
                float sum[128];
#pragma unroll 1
                for (int j = 0; j < kKSplitSlices; ++j) {
                    const int q = 2 * (job++ & 1);
                    if (!wait_full(q)) {
                        go = false;
                        break;
                    }
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        uint32_t u[16];
                        ptx::tmem_ld_x16(acc0 + (uint32_t)(128 * q + 16 * ch), u);
                        ptx::tmem_ld_wait();
                        if (ch == 7) {
                            release(q);
                            release(q + 1);
                        }
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float p = bf16_round(__uint_as_float(u[e]));
                            sum[16 * ch + e] = j == 0 ? p : sum[16 * ch + e] + p;
                        }
                    }
                }
                if (!go) break;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t v[16];
                    const int y = row0 + 128 * cs + 16 * ch;
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) v[jj] = bf16_bits(sum[16 * ch + jj]);
                    store_chunk(v, false, &map_lat, xw, y, valid);
                    if (args.ss_part != nullptr) sumsq_parts(part, y, std::false_type{});
                }
            }
        }
        if (lane == 0) ptx::bulk_wait_group_all();  // every store has left shared memory
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // the leader's MMAs write this CTA's TMEM: the peer waits for them too
        if (lane == 0 && !leader) wait_drain(drain_bar, 0u, args);
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
    }
    ptx::cluster_sync();  // neither CTA leaves while the other may reach its shared memory
}

}  // namespace

int prefill_smem_bytes() { return (int)kSmemBytes; }

cudaError_t prefill_configure() {
    return cudaFuncSetAttribute(prefill_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemBytes);
}

cudaError_t prefill_launch(const CUtensorMap &map_h, const CUtensorMap &map_wl,
                           const CUtensorMap &map_wr, const CUtensorMap &map_lat,
                           const CUtensorMap &map_lg, const ProjArgs &args, cudaStream_t stream) {
    if (args.grid <= 0 || args.grid % 2 != 0) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t c = {};
    cudaLaunchAttribute attr[1];
    c.gridDim = dim3(args.grid);
    c.blockDim = dim3(kProjThreads);
    c.dynamicSmemBytes = kSmemBytes;
    c.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    c.attrs = attr;
    c.numAttrs = 1;
    return cudaLaunchKernelEx(&c, prefill_pair_kernel, map_h, map_wl, map_wr, map_lat, map_lg, args);
}

}  // namespace route
