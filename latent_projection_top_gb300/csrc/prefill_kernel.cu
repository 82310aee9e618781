// Prefill route projection (steps a1 and a2 for a chunk of token rows) on
// the sm_103a tensor cores, two SMs per tile.
//
//   latent[r, n] = bf16( sum_k hidden[r, k] * W_latent[k, n] )   n < 3584
//   logits[r, e] =       sum_k hidden[r, k] * W_router[k, e]    e < 896
//
// Each output is one FP32-accumulated dot product over the full K = 7168,
// rounded once ("Optionally gather the Kimi3 prefill latent instead of
// reducing it", Description, Numerics and Compile bullets: at prefill the
// projection is a dense M = rows, K = 7168 GEMM); the two projections share
// the hidden operand and run as one N = 3584 + 896 problem.
//
// The weights are [K, N] with N contiguous, so their tensor-core operand is
// MN-major.  A tile is 256 weight columns (the MMA's M) by 256 token rows
// (its N), computed by a cluster of two CTAs with tcgen05.mma.cta_group::2:
// each CTA stages its half of the weight columns (A, 128 x 64 per k-block)
// and its half of the token rows (B, 128 x 64), and holds its 128 weight
// columns x 256 token rows of the FP32 accumulator in its own TMEM.  Against
// one CTA per 128 x 256 tile this moves a third fewer bytes from L2 per
// flop and leaves room for a 6-stage ring.
//
// Warp roles (192 threads, persistent, one CTA per SM, pairs = clusters):
//   warp 0      TMA producer (both CTAs): its halves into a 6-stage ring;
//               completion is counted on the leader CTA's barrier, which the
//               leader arms for both CTAs' bytes before either may fill the
//               stage (so its transaction count never goes below zero)
//   warp 1      TMEM owner (both CTAs); the leader's lane 0 issues the MMAs
//               and re-arms each stage's barrier once it has consumed it
//   warps 2..5  epilogue (both CTAs): TMEM -> registers -> global
// Pairs walk the (row tile, column tile) grid with stride = number of pairs;
// two TMEM accumulators let one tile's epilogue overlap the next main loop.
//
// With the general path's K-split latent (args.ksplit), a latent tile runs as
// eight jobs of 14 k-blocks into one accumulator; the epilogue rounds each
// slice's partial to BF16 and adds it in FP32 to a running sum kept in the
// other half of TMEM, rounding and storing after the eighth.
//
// Programmatic dependent launch: weight boxes of the first stages are
// requested before `griddepcontrol.wait` (no predecessor writes the weights);
// outputs are written only after it, and hidden rows are read only after it
// too unless `overlap` is set (then the main loop runs under the previous
// step's top-16).
//
// Every wait is bounded: after args.timeout_ns a waiting thread sets the
// device status word and the CTA's abort flag, in-flight copies and MMAs are
// drained, TMEM is freed and the CTA returns (both CTAs of a pair meet at a
// final cluster barrier, so neither leaves while the other may still reach
// its shared memory).
#include <cuda_bf16.h>

#include "common.cuh"
#include "sm103_ptx.cuh"

namespace route {
namespace {

constexpr uint32_t kABoxBytes = 64 * 64 * 2;               // 64 columns x 64 k, BF16
constexpr int kHalf = 128;                                 // each CTA's share of M and of N
constexpr int kPairCols = 2 * kHalf;                       // weight columns per tile (M)
constexpr int kPairRows = kPrefillBN;                      // token rows per tile (N)
constexpr uint32_t kBHalfBytes = kHalf * 128;              // 128 token rows x 64 k
constexpr uint32_t kAHalfBytes = 2 * kABoxBytes;           // 128 weight columns x 64 k
constexpr uint32_t kStageBytes = kBHalfBytes + kAHalfBytes;  // B half first, then A half
constexpr int kStages = 6;
constexpr uint32_t kSmemBytes = 1024 + kStages * kStageBytes + 256;
constexpr uint32_t kTmemCols = 512;                        // two accumulators of 256 columns
constexpr int kLatPairTiles = kLatent / kPairCols;         // 14
constexpr int kPairColTiles = kLatPairTiles + (kExperts + kPairCols - 1) / kPairCols;  // 18
// tcgen05 instruction descriptor, kind::f16: FP32 accumulator, BF16 A and B,
// A MN-major (transposed), B K-major, N = 256, M = 256 (over the pair).
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) |
                            ((uint32_t)(kPairRows >> 3) << 17) | ((uint32_t)(kPairCols >> 4) << 24);
static_assert(kPairColTiles == kPrefillColTiles, "column tiles");
static_assert(kHalf == kPrefillHiddenBoxRows, "hidden box");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
static_assert(8 * (2 * kStages + 5) <= 256, "barrier area");
static_assert(kLatent % kPairCols == 0, "latent tiles");

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

struct Tile {
    int c;   // column tile: 0..13 latent, 14..17 router (the last has 128 real columns)
    int rt;  // row tile
};

__device__ __forceinline__ int tiles_of_pair(const ProjArgs &a, int pair, int npairs) {
    const int tiles = kPairColTiles * a.row_tiles;
    return pair < tiles ? (tiles - 1 - pair) / npairs + 1 : 0;
}

// Tiles in row-major order: the pairs at work at one time share a few
// 256-row blocks of hidden and read every weight tile (measured 117 us
// against 128 us at 3072 rows for column-major order).
__device__ __forceinline__ Tile tile_get(const ProjArgs &a, int pair, int npairs, int i) {
    const int t = pair + i * npairs;
    return Tile{t % kPairColTiles, t / kPairColTiles};
}

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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kProjThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap map_h,
                        const __grid_constant__ CUtensorMap map_wl,
                        const __grid_constant__ CUtensorMap map_wr,
                        const __grid_constant__ ProjArgs args) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem_base;
    __shared__ volatile int s_abort;

    // Both CTAs of a pair lay out shared memory identically, so an offset in
    // one names the same operand or barrier in the other.
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    const uint32_t bars = sbase + kStages * kStageBytes;
    auto full_bar = [&](int s) { return bars + 8u * s; };                 // leader's are used
    auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
    auto accfull_bar = [&](int b) { return bars + 8u * (2 * kStages + b); };
    auto accempty_bar = [&](int b) { return bars + 8u * (2 * kStages + 2 + b); };  // leader's
    const uint32_t drain_bar = bars + 8u * (2 * kStages + 4);

    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = rank == 0u;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;
    const int nseg = tiles_of_pair(args, pair, npairs);

    if (threadIdx.x == 0) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        s_abort = 0;
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accfull_bar(b), 1);
            ptx::mbar_init(accempty_bar(b), 2);  // one arrival from each CTA's epilogue
        }
        ptx::mbar_init(drain_bar, 1);
        // the leader arms the first round of every stage that will be filled
        const int first = nseg * kKBlocks < kStages ? nseg * kKBlocks : kStages;
        if (leader)
            for (int s = 0; s < first; ++s) ptx::mbar_arrive_expect_tx(full_bar(s), 2 * kStageBytes);
        ptx::fence_barrier_init();
        ptx::prefetch_tensormap(&map_h);
        ptx::prefetch_tensormap(&map_wl);
        ptx::prefetch_tensormap(&map_wr);
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
            const uint64_t pol_w = ptx::policy_evict_normal();
            const uint64_t pol_h = ptx::policy_evict_last();
            uint32_t armed = 0u, armed_par = 0u;  // leader: stages armed / their phase parity
            const int total = nseg * kKBlocks;
            const int n_pre = total < kStages ? total : kStages;
            auto weights_of = [&](int it, uint32_t st, uint32_t bar) {
                const Tile tl = tile_get(args, pair, npairs, it / kKBlocks);
                const int kb = it % kKBlocks;
                const bool lat = tl.c < kLatPairTiles;
                const CUtensorMap *wmap = lat ? &map_wl : &map_wr;
                // this CTA's 128 columns; past column 896 of W_router TMA fills zeros
                const int x0 = (lat ? tl.c : tl.c - kLatPairTiles) * kPairCols + (int)rank * kHalf;
                ptx::tma_load_2d_pair(st + kBHalfBytes, wmap, bar, x0, kb * kKBlock, pol_w);
                ptx::tma_load_2d_pair(st + kBHalfBytes + kABoxBytes, wmap, bar, x0 + 64,
                                      kb * kKBlock, pol_w);
            };
            auto hidden_of = [&](int it, uint32_t st, uint32_t bar) {
                const Tile tl = tile_get(args, pair, npairs, it / kKBlocks);
                ptx::tma_load_2d_pair(st, &map_h, bar, (it % kKBlocks) * kKBlock,
                                      tl.rt * kPairRows + (int)rank * kHalf, pol_h);
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
            uint32_t it = 0, job = 0;
            bool ok = true;
            for (int i = 0; i < nseg && ok; ++i) {
                const Tile tl = tile_get(args, pair, npairs, i);
                const int njobs = (args.ksplit && tl.c < kLatPairTiles) ? kKSplitSlices : 1;
                const int kb_per_job = kKBlocks / njobs;
                for (int j = 0; j < njobs && ok; ++j, ++job) {
                    const int buf = args.ksplit ? 0 : (int)(job & 1u);
                    const uint32_t use = args.ksplit ? job : (job >> 1);
                    if (!wait_phase(accempty_bar(buf), (use & 1u) ^ 1u, args, &s_abort)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (uint32_t)(buf * kPairRows);
                    for (int kb = 0; kb < kb_per_job; ++kb, ++it) {
                        const int s = (int)(it % kStages);
                        const uint32_t ph = (it / kStages) & 1u;
                        if (!wait_phase(full_bar(s), ph, args, &s_abort)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t b = sbase + s * kStageBytes;
                        const uint32_t a = b + kBHalfBytes;
#pragma unroll
                        for (int kk = 0; kk < kKBlock / 16; ++kk) {
                            // A: k advances 16 rows = two 8-row swizzle atoms (2048 B);
                            //    the two 64-column boxes are 8192 B apart (LBO),
                            //    8-row k groups 1024 B apart (SBO).
                            // B: k advances 32 B inside the 128-byte swizzled row;
                            //    8-row groups of token rows are 1024 B apart (SBO).
                            const uint64_t da = smem_desc(a + kk * 2048u, kABoxBytes, 1024u);
                            const uint64_t db = smem_desc(b + kk * 32u, 16u, 1024u);
                            ptx::mma_bf16_pair(d_tmem, da, db, kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
                        }
                        // re-arm stage s for its next round before it is freed:
                        // the copies that fill it can only start after the commit
                        if (it + kStages < (uint32_t)(nseg * kKBlocks))
                            ptx::mbar_arrive_expect_tx(full_bar(s), 2 * kStageBytes);
                        ptx::mma_commit_pair(empty_bar(s), 0x3);  // frees stage s in both CTAs
                    }
                    if (ok) ptx::mma_commit_pair(accfull_bar(buf), 0x3);
                }
            }
            ptx::mma_commit_pair(drain_bar, 0x3);  // every MMA retired before TMEM is freed
            wait_drain(drain_bar, 0u, args);
        }
    } else {
        // ---------------- epilogue (warps 2..5, both CTAs) ----------------
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
        const int col = 32 * quarter + lane;
        const int rows = args.rows;
        asm volatile("griddepcontrol.wait;" ::: "memory");  // outputs may still be read by the predecessor
        uint32_t job = 0;
        bool go = true;
        for (int i = 0; i < nseg && go; ++i) {
            const Tile tl = tile_get(args, pair, npairs, i);
            const bool lat = tl.c < kLatPairTiles;
            const int njobs = (args.ksplit && lat) ? kKSplitSlices : 1;
            const int ncol = (lat ? tl.c : tl.c - kLatPairTiles) * kPairCols + (int)rank * kHalf + col;
            const bool valid = lat || ncol < kExperts;
            for (int j = 0; j < njobs; ++j, ++job) {
                const int buf = args.ksplit ? 0 : (int)(job & 1u);
                const uint32_t use = args.ksplit ? job : (job >> 1);
                const bool ok = wait_phase(accfull_bar(buf), use & 1u, args, &s_abort);
                if (!ptx::named_bar_and(1, 128, ok)) {
                    go = false;
                    break;
                }
                __syncwarp();  // the TMEM loads below are warp-wide (.sync.aligned)
                ptx::tc_fence_after();
                const uint32_t lanes = tmem_base + ((uint32_t)(32 * quarter) << 16);
                const uint32_t taddr = lanes + (uint32_t)(buf * kPairRows);
                if (njobs == 1) {
#pragma unroll 1
                    for (int ch = 0; ch < kPairRows / 16; ++ch) {
                        uint32_t u[16];
                        ptx::tmem_ld_x16(taddr + ch * 16, u);
                        ptx::tmem_ld_wait();
                        const int r0 = tl.rt * kPairRows + ch * 16;
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int r = r0 + jj;
                            if (valid && r < rows) {
                                const float x = __uint_as_float(u[jj]);
                                if (lat)
                                    args.latent[(size_t)r * kLatent + ncol] = bf16_bits(x);
                                else
                                    args.logits[(size_t)r * kExperts + ncol] = x;
                            }
                        }
                    }
                } else {
                    // K-split latent: slice j's partial, rounded to BF16, is
                    // added in FP32 to the running sum kept in the other half
                    // of TMEM; the last slice rounds the sum to BF16 and stores.
                    const uint32_t tsum = lanes + (uint32_t)kPairRows;
                    const bool last = j == njobs - 1;
#pragma unroll 1
                    for (int ch = 0; ch < kPairRows / 16; ++ch) {
                        uint32_t u[16], acc[16];
                        ptx::tmem_ld_x16(taddr + ch * 16, u);
                        if (j > 0) ptx::tmem_ld_x16(tsum + ch * 16, acc);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const float part = __uint_as_float((uint32_t)bf16_bits(__uint_as_float(u[jj])) << 16);
                            acc[jj] = __float_as_uint(j > 0 ? __uint_as_float(acc[jj]) + part : part);
                        }
                        if (!last) {
                            ptx::tmem_st_x16(tsum + ch * 16, acc);
                        } else {
                            const int r0 = tl.rt * kPairRows + ch * 16;
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj)
                                if (r0 + jj < rows)
                                    args.latent[(size_t)(r0 + jj) * kLatent + ncol] =
                                        bf16_bits(__uint_as_float(acc[jj]));
                        }
                    }
                    if (!last) ptx::tmem_st_wait();  // the next slice reads these sums back
                }
                // all 128 epilogue threads are done with this accumulator: one
                // arrival from this CTA on the leader's barrier
                ptx::tc_fence_before();
                ptx::named_bar_sync(2, 128);
                if (threadIdx.x == 64) {
                    if (leader)
                        ptx::mbar_arrive(accempty_bar(buf));
                    else
                        ptx::mbar_arrive_remote(ptx::map_to_rank(accempty_bar(buf), 0u));
                }
            }
        }
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
                           const CUtensorMap &map_wr, const ProjArgs &args, cudaStream_t stream) {
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
    return cudaLaunchKernelEx(&c, prefill_pair_kernel, map_h, map_wl, map_wr, args);
}

}  // namespace route
