// Prefill route projection (steps a1 and a2 for a chunk of token rows) on
// the sm_103a tensor cores.
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
// MN-major.  A tile is 128 weight columns on the MMA M side (A = W^T, two
// 64x64 TMA boxes per k-block) by 256 token rows on the N side (B = hidden,
// K-major), accumulated in TMEM over all 112 k-blocks.
//
// Warp roles (192 threads, persistent, one CTA per SM):
//   warp 0      TMA producer: weight + hidden boxes into a 4-stage smem ring
//   warp 1      TMEM owner and single-thread tcgen05.mma issuer
//   warps 2..5  epilogue: TMEM -> registers -> global (one TMEM lane quarter each)
// CTAs walk the (column tile, row tile) grid with stride gridDim; two TMEM
// accumulators let one tile's epilogue overlap the next tile's main loop.
//
// Programmatic dependent launch: weight boxes of the first stages are
// requested before `griddepcontrol.wait` (no predecessor writes the weights);
// hidden rows are read and outputs written only after it.
//
// Every wait is bounded: after args.timeout_ns a waiting thread sets the
// device status word and the CTA's abort flag, in-flight copies and MMAs are
// drained, TMEM is freed and the CTA returns.
#include <cuda_bf16.h>

#include "common.cuh"
#include "sm103_ptx.cuh"

namespace route {
namespace {

constexpr uint32_t kABoxBytes = 64 * 64 * 2;       // 64 columns x 64 k, BF16
constexpr uint32_t kAStageBytes = 2 * kABoxBytes;  // 128 columns x 64 k

template <int BN>
struct ProjCfg {
    static constexpr uint32_t kBStageBytes = BN * 128;  // BN rows x 64 k, BF16
    static constexpr uint32_t kStageBytes = kAStageBytes + kBStageBytes;
    static constexpr int kStages = BN >= 256 ? 4 : 10;
    static constexpr uint32_t kTmemCols = 2 * BN <= 32    ? 32
                                          : 2 * BN <= 64  ? 64
                                          : 2 * BN <= 128 ? 128
                                          : 2 * BN <= 256 ? 256
                                                          : 512;
    static constexpr uint32_t kSmemBytes = 1024 + kStages * kStageBytes + 256;
    // tcgen05 instruction descriptor, kind::f16: FP32 accumulator, BF16 A and
    // B, A MN-major (transposed), B K-major, N = BN, M = 128.
    static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) |
                                       ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M = 128");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
    static_assert(2 * kStages + 5 <= 32, "barrier area");
};

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

struct Seg {
    int c;   // column tile (0..27 latent, 28..34 router)
    int rt;  // row tile
};

__device__ __forceinline__ int seg_total(const ProjArgs &a, int g) {
    const int tiles = kColTiles * a.row_tiles;
    return g < tiles ? (tiles - 1 - g) / a.grid + 1 : 0;
}

__device__ __forceinline__ Seg seg_get(const ProjArgs &a, int g, int i) {
    const int t = g + i * a.grid;
    return Seg{t / a.row_tiles, t % a.row_tiles};
}

// Bounded wait for the completion of phase `parity` of `bar`.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const ProjArgs &a,
                                           volatile int *abort_flag) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
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

// Bounded wait used only while tearing down after an abort.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, const ProjArgs &a) {
    const uint64_t t0 = ptx::global_timer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::global_timer_ns() - t0 > a.timeout_ns) {
            atomicOr(a.status, kStatusTimeout);
            return;
        }
    }
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

template <int BN>
__global__ void __launch_bounds__(kProjThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_wl,
                   const __grid_constant__ CUtensorMap map_wr, const __grid_constant__ ProjArgs args) {
    using C = ProjCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem_base;
    __shared__ volatile int s_abort;

    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    const uint32_t bars = sbase + C::kStages * C::kStageBytes;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (C::kStages + s); };
    auto accfull_bar = [&](int b) { return bars + 8u * (2 * C::kStages + b); };
    auto accempty_bar = [&](int b) { return bars + 8u * (2 * C::kStages + 2 + b); };
    const uint32_t drain_bar = bars + 8u * (2 * C::kStages + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = blockIdx.x;
    const int nseg = seg_total(args, g);

    if (threadIdx.x == 0) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        s_abort = 0;
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accfull_bar(b), 1);
            ptx::mbar_init(accempty_bar(b), 128);
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
            const uint64_t pol_w = ptx::policy_evict_normal();
            const uint64_t pol_h = ptx::policy_evict_last();
            uint32_t armed = 0u, armed_par = 0u;  // per stage: loads issued / their phase parity
            const int total = nseg * kKBlocks;
            const int n_pre = total < C::kStages ? total : C::kStages;
            auto weights_of = [&](int it, uint32_t a, uint32_t bar) {
                const Seg sg = seg_get(args, g, it / kKBlocks);
                const int kb = it % kKBlocks;
                const bool lat = sg.c < kLatentTiles;
                const CUtensorMap *wmap = lat ? &map_wl : &map_wr;
                const int x0 = (lat ? sg.c : sg.c - kLatentTiles) * kTileCols;
                ptx::tma_load_2d(a, wmap, bar, x0, kb * kKBlock, pol_w);
                ptx::tma_load_2d(a + kABoxBytes, wmap, bar, x0 + 64, kb * kKBlock, pol_w);
            };
            auto hidden_of = [&](int it, uint32_t a, uint32_t bar) {
                const Seg sg = seg_get(args, g, it / kKBlocks);
                ptx::tma_load_2d(a + kAStageBytes, &map_h, bar, (it % kKBlocks) * kKBlock, sg.rt * BN,
                                 pol_h);
            };
            // Weight boxes of the first stages go out before the grid
            // dependency resolves (no predecessor writes the weights).
            for (int it = 0; it < n_pre; ++it) {
                ptx::mbar_arrive_expect_tx(full_bar(it), C::kStageBytes);
                weights_of(it, sbase + it * C::kStageBytes, full_bar(it));
                armed |= 1u << it;
            }
            asm volatile("griddepcontrol.wait;" ::: "memory");
            for (int it = 0; it < n_pre; ++it) {
                if (args.test_stall && it == total - 1) continue;  // test hook
                hidden_of(it, sbase + it * C::kStageBytes, full_bar(it));
            }
            bool ok = true;
            for (int it = n_pre; it < total; ++it) {
                const int s = it % C::kStages;
                const uint32_t ph = (uint32_t)(it / C::kStages) & 1u;
                if (!wait_phase(empty_bar(s), ph ^ 1u, args, &s_abort)) {
                    ok = false;
                    break;
                }
                if (args.test_stall && it == total - 1) continue;  // test hook: never filled
                const uint32_t a = sbase + s * C::kStageBytes;
                ptx::mbar_arrive_expect_tx(full_bar(s), C::kStageBytes);
                weights_of(it, a, full_bar(s));
                hidden_of(it, a, full_bar(s));
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
            // ---------------- MMA issuer ----------------
            uint32_t it = 0;
            bool ok = true;
            for (int i = 0; i < nseg && ok; ++i) {
                const int buf = i & 1;
                const uint32_t use = (uint32_t)(i >> 1);
                if (!wait_phase(accempty_bar(buf), (use & 1u) ^ 1u, args, &s_abort)) break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
                for (int kb = 0; kb < kKBlocks; ++kb, ++it) {
                    const int s = (int)(it % C::kStages);
                    const uint32_t ph = (it / C::kStages) & 1u;
                    if (!wait_phase(full_bar(s), ph, args, &s_abort)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a = sbase + s * C::kStageBytes;
                    const uint32_t b = a + kAStageBytes;
#pragma unroll
                    for (int kk = 0; kk < kKBlock / 16; ++kk) {
                        // A: k advances 16 rows = two 8-row swizzle atoms (2048 B);
                        //    the two 64-column boxes are 8192 B apart (LBO),
                        //    8-row k groups 1024 B apart (SBO).
                        // B: k advances 32 B inside the 128-byte swizzled row;
                        //    8-row groups of token rows are 1024 B apart (SBO).
                        const uint64_t da = smem_desc(a + kk * 2048u, kABoxBytes, 1024u);
                        const uint64_t db = smem_desc(b + kk * 32u, 16u, 1024u);
                        ptx::mma_bf16(d_tmem, da, db, C::kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit(empty_bar(s));
                }
                if (ok) ptx::mma_commit(accfull_bar(buf));
            }
            ptx::mma_commit(drain_bar);  // every MMA retired before TMEM is freed
            wait_drain(drain_bar, 0u, args);
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
        const int col = 32 * quarter + lane;
        const int rows = args.rows;
        asm volatile("griddepcontrol.wait;" ::: "memory");  // outputs may still be read by the predecessor
        for (int i = 0; i < nseg; ++i) {
            const Seg sg = seg_get(args, g, i);
            const int buf = i & 1;
            const uint32_t use = (uint32_t)(i >> 1);
            const bool ok = wait_phase(accfull_bar(buf), use & 1u, args, &s_abort);
            if (!ptx::named_bar_and(1, 128, ok)) break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(buf * BN);
            const bool lat = sg.c < kLatentTiles;
            const int ncol = (lat ? sg.c : sg.c - kLatentTiles) * kTileCols + col;
#pragma unroll 1
            for (int ch = 0; ch < BN / 16; ++ch) {
                uint32_t u[16];
                ptx::tmem_ld_x16(taddr + ch * 16, u);
                ptx::tmem_ld_wait();
                const int r0 = sg.rt * BN + ch * 16;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int r = r0 + j;
                    if (r < rows) {
                        const float x = __uint_as_float(u[j]);
                        if (lat)
                            args.latent[(size_t)r * kLatent + ncol] = bf16_bits(x);
                        else
                            args.logits[(size_t)r * kExperts + ncol] = x;
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(accempty_bar(buf));
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

}  // namespace

int prefill_smem_bytes() { return (int)ProjCfg<kPrefillBN>::kSmemBytes; }

cudaError_t prefill_configure() {
    return cudaFuncSetAttribute(prefill_kernel<kPrefillBN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)ProjCfg<kPrefillBN>::kSmemBytes);
}

cudaError_t prefill_launch(const CUtensorMap &map_h, const CUtensorMap &map_wl,
                           const CUtensorMap &map_wr, const ProjArgs &args, cudaStream_t stream) {
    cudaLaunchConfig_t c = {};
    cudaLaunchAttribute attr[1];
    c.gridDim = dim3(args.grid);
    c.blockDim = dim3(kProjThreads);
    c.dynamicSmemBytes = ProjCfg<kPrefillBN>::kSmemBytes;
    c.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    c.attrs = attr;
    c.numAttrs = 1;
    return cudaLaunchKernelEx(&c, prefill_kernel<kPrefillBN>, map_h, map_wl, map_wr, args);
}

}  // namespace route
