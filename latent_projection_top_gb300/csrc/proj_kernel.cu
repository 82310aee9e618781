// Latent down projection + router logits (route-step steps a1 and a2) on the
// sm_103a tensor cores.
//
//   latent[r, n] = bf16( sum_k hidden[r, k] * W_latent[k, n] )   n < 3584
//   logits[r, e] =       sum_k hidden[r, k] * W_router[k, e]    e < 896
//
// Each output is one FP32-accumulated dot product over the full K = 7168,
// rounded once ("Optionally gather the Kimi3 prefill latent instead of
// reducing it", Description, Numerics bullet); the two projections share the
// hidden operand and run as one N = 3584 + 896 problem.
//
// The weights are [K, N] with N contiguous, so the tensor-core operand that
// comes from them is MN-major.  The kernel puts 128 weight columns on the MMA
// M side (A = W^T tile, MN-major, from two 64x64 TMA boxes) and BN token rows
// on the N side (B = hidden tile, K-major), accumulating D^T[col, row] in TMEM.
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: weight + hidden boxes into a ring of smem stages
//   warp 1      TMEM owner and single-thread tcgen05.mma issuer
//   warps 2..5  epilogue: TMEM -> registers -> global (one TMEM lane quarter each)
//
// Two schedules over the same kernel:
//   decode  (1..20 rows, BN = 16 or 32): HBM-bound weight streaming.  The
//           35 x 112 (column tile, k-block) units are cut into equal
//           contiguous ranges, one per CTA; a CTA's range touches one or two
//           column tiles.  Each piece ("segment") leaves an FP32 partial in
//           scratch; the CTA that arrives last at a tile (atomic counter) sums
//           the tile's partials in segment order, rounds once and writes.  The
//           partition depends only on the grid, so results are reproducible
//           and a row's bits do not depend on the number of rows.  With
//           fuse_topk, the CTA that completes the last router tile runs the
//           top-16 for every row (the whole route step in one launch).
//   prefill (BN = 256): persistent CTAs walk (column tile, row tile) tiles
//           with the full K each; two TMEM accumulators let the epilogue of
//           one tile overlap the main loop of the next.
//
// Every wait is bounded: after args.timeout_ns a waiting thread sets the
// device status word and the CTA's abort flag, in-flight copies and MMAs are
// drained, TMEM is freed and the CTA returns.
#include <cuda_bf16.h>

#include "common.cuh"
#include "sm103_ptx.cuh"
#include "topk16.cuh"

namespace route {
namespace {

constexpr uint32_t kABoxBytes = 64 * 64 * 2;       // 64 columns x 64 k, BF16
constexpr uint32_t kAStageBytes = 2 * kABoxBytes;  // 128 columns x 64 k
constexpr int kReduceBatch = 8;                    // split-K partials loaded per batch

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
    int c;     // column tile (0..27 latent, 28..34 router)
    int rt;    // row tile
    int kb0;   // first k-block
    int kb1;   // one past the last k-block
    int slot;  // decode: partial slot in scratch
};

__device__ __forceinline__ long long unit_lo(const ProjArgs &a, int g) {
    return (long long)g * a.units / a.grid;
}

__device__ __forceinline__ int seg_total(const ProjArgs &a, int g) {
    if (a.mode == kDecode) {
        long long u0 = unit_lo(a, g), u1 = unit_lo(a, g + 1);
        if (u1 <= u0) return 0;
        return (int)((u1 - 1) / kKBlocks - u0 / kKBlocks + 1);
    }
    int tiles = kColTiles * a.row_tiles;
    return g < tiles ? (tiles - 1 - g) / a.grid + 1 : 0;
}

__device__ __forceinline__ Seg seg_get(const ProjArgs &a, int g, int i) {
    Seg s;
    if (a.mode == kDecode) {
        long long u0 = unit_lo(a, g), u1 = unit_lo(a, g + 1);
        s.c = (int)(u0 / kKBlocks) + i;
        long long lo = u0 > (long long)s.c * kKBlocks ? u0 : (long long)s.c * kKBlocks;
        long long hi = u1 < (long long)(s.c + 1) * kKBlocks ? u1 : (long long)(s.c + 1) * kKBlocks;
        s.kb0 = (int)(lo - (long long)s.c * kKBlocks);
        s.kb1 = (int)(hi - (long long)s.c * kKBlocks);
        s.rt = 0;
        s.slot = a.seg_base[s.c] + (g - a.cta_first[s.c]);
    } else {
        int t = g + i * a.grid;
        s.c = t / a.row_tiles;
        s.rt = t % a.row_tiles;
        s.kb0 = 0;
        s.kb1 = kKBlocks;
        s.slot = -1;
    }
    return s;
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
    proj_kernel(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_wl,
                const __grid_constant__ CUtensorMap map_wr, const __grid_constant__ ProjArgs args) {
    using C = ProjCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem_base;
    __shared__ volatile int s_abort;
    __shared__ int s_last;
    __shared__ uint2 s_cand[4][kCandMax];  // fused top-16 candidates, one buffer per epilogue warp

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
            const uint64_t pol_w =
                args.mode == kDecode ? ptx::policy_evict_first() : ptx::policy_evict_normal();
            const uint64_t pol_h = ptx::policy_evict_last();
            uint32_t armed = 0u, armed_par = 0u;  // per stage: loads issued / their phase parity
            uint32_t it = 0;
            bool ok = true;
            for (int i = 0; i < nseg && ok; ++i) {
                const Seg sg = seg_get(args, g, i);
                const bool lat = sg.c < kLatentTiles;
                const CUtensorMap *wmap = lat ? &map_wl : &map_wr;
                const int x0 = (lat ? sg.c : sg.c - kLatentTiles) * kTileCols;
                for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
                    const int s = (int)(it % C::kStages);
                    const uint32_t ph = (it / C::kStages) & 1u;
                    if (!wait_phase(empty_bar(s), ph ^ 1u, args, &s_abort)) {
                        ok = false;
                        break;
                    }
                    if (args.test_stall && i == nseg - 1 && kb == sg.kb1 - 1)
                        continue;  // test hook: this stage is never filled
                    const uint32_t a = sbase + s * C::kStageBytes;
                    ptx::mbar_arrive_expect_tx(full_bar(s), C::kStageBytes);
                    ptx::tma_load_2d(a, wmap, full_bar(s), x0, kb * kKBlock, pol_w);
                    ptx::tma_load_2d(a + kABoxBytes, wmap, full_bar(s), x0 + 64, kb * kKBlock, pol_w);
                    ptx::tma_load_2d(a + kAStageBytes, &map_h, full_bar(s), kb * kKBlock, sg.rt * BN,
                                     pol_h);
                    armed |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                }
            }
            if (!ok) {  // let every issued copy land before the CTA may exit
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
                const Seg sg = seg_get(args, g, i);
                const int buf = i & 1;
                const uint32_t use = (uint32_t)(i >> 1);
                if (!wait_phase(accempty_bar(buf), (use & 1u) ^ 1u, args, &s_abort)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
                for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
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
                        ptx::mma_bf16(d_tmem, da, db, C::kIdesc, (kb > sg.kb0 || kk > 0) ? 1u : 0u);
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
        const int et = threadIdx.x - 64;
        const int rows = args.rows;
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

            if constexpr (BN <= 32) {
                // decode schedule (the host only pairs BN <= 32 with decode)
                float v[BN];
#pragma unroll
                for (int ch = 0; ch < BN / 16; ++ch) {
                    uint32_t u[16];
                    ptx::tmem_ld_x16(taddr + ch * 16, u);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[ch * 16 + j] = __uint_as_float(u[j]);
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(accempty_bar(buf));

                float *part = args.ws + (size_t)sg.slot * kDecodeMaxRows * kTileCols + col;
#pragma unroll
                for (int r = 0; r < BN; ++r)
                    if (r < rows) part[r * kTileCols] = v[r];
                __threadfence();
                ptx::named_bar_sync(1, 128);
                if (et == 0) {
                    const unsigned prev = atomicAdd(&args.counters[sg.c], 1u);
                    s_last = (prev == (unsigned)(args.seg_count[sg.c] - 1));
                }
                ptx::named_bar_sync(1, 128);
                if (s_last) {
                    // Last arrival: sum the tile's partials in segment order.
                    // Items are (row, 4 columns); all of an item's partials are
                    // loaded before any is added, two items at a time.
                    __threadfence();
                    const int ns = args.seg_count[sg.c];
                    const float *p0 = args.ws + (size_t)args.seg_base[sg.c] * kDecodeMaxRows * kTileCols;
                    const int items = rows * (kTileCols / 4);
                    const int nbase = (lat ? sg.c : sg.c - kLatentTiles) * kTileCols;
                    for (int it0 = et; it0 < items; it0 += 256) {
                        float4 acc[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                        for (int s0 = 0; s0 < ns; s0 += kReduceBatch) {
                            float4 part[2][kReduceBatch];
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const int it = it0 + 128 * u;
                                const float *p = p0 + (it >> 5) * kTileCols + (it & 31) * 4;
#pragma unroll
                                for (int j = 0; j < kReduceBatch; ++j)
                                    if (it < items && s0 + j < ns)
                                        part[u][j] = __ldcg(reinterpret_cast<const float4 *>(
                                            p + (size_t)(s0 + j) * kDecodeMaxRows * kTileCols));
                            }
#pragma unroll
                            for (int u = 0; u < 2; ++u)
#pragma unroll
                                for (int j = 0; j < kReduceBatch; ++j)
                                    if (s0 + j < ns) {
                                        if (s0 + j == 0) {
                                            acc[u] = part[u][j];
                                        } else {
                                            acc[u].x += part[u][j].x;
                                            acc[u].y += part[u][j].y;
                                            acc[u].z += part[u][j].z;
                                            acc[u].w += part[u][j].w;
                                        }
                                    }
                        }
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int it = it0 + 128 * u;
                            if (it >= items) continue;
                            const int r = it >> 5;
                            const int n = nbase + (it & 31) * 4;
                            if (lat) {
                                uint2 packed;
                                packed.x = (uint32_t)bf16_bits(acc[u].x) | ((uint32_t)bf16_bits(acc[u].y) << 16);
                                packed.y = (uint32_t)bf16_bits(acc[u].z) | ((uint32_t)bf16_bits(acc[u].w) << 16);
                                *reinterpret_cast<uint2 *>(args.latent + (size_t)r * kLatent + n) = packed;
                            } else {
                                *reinterpret_cast<float4 *>(args.logits + (size_t)r * kExperts + n) = acc[u];
                            }
                        }
                    }
                    if (et == 0) args.counters[sg.c] = 0u;  // ready for the next launch
                    if (args.fuse_topk && !lat) {
                        __threadfence();
                        ptx::named_bar_sync(1, 128);
                        if (et == 0) {
                            const unsigned prev = atomicAdd(&args.counters[kColTiles], 1u);
                            s_last = (prev == (unsigned)(kRouterTiles - 1));
                        }
                        ptx::named_bar_sync(1, 128);
                        if (s_last) {
                            // Every router tile is final: run the top-16 for all rows.
                            __threadfence();
                            for (int r = et >> 5; r < rows; r += 4)
                                topk16_warp(args.logits + (size_t)r * kExperts,
                                            args.ids + (size_t)r * kTopK,
                                            args.weights + (size_t)r * kTopK, lane,
                                            s_cand[et >> 5]);
                            if (et == 0) args.counters[kColTiles] = 0u;
                        }
                    }
                }
            } else {
                // prefill schedule: full-K tile straight to the outputs
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
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

template <int BN>
cudaError_t configure_bn() {
    return cudaFuncSetAttribute(proj_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)ProjCfg<BN>::kSmemBytes);
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap &mh, const CUtensorMap &ml, const CUtensorMap &mr,
                      const ProjArgs &args, cudaStream_t stream) {
    proj_kernel<BN><<<args.grid, kProjThreads, ProjCfg<BN>::kSmemBytes, stream>>>(mh, ml, mr, args);
    return cudaGetLastError();
}

}  // namespace

int proj_bn_for(int mode, int rows) {
    if (mode == kPrefill) return 256;
    return rows <= 16 ? 16 : 32;
}

int proj_smem_bytes(int bn) {
    switch (bn) {
        case 16: return (int)ProjCfg<16>::kSmemBytes;
        case 32: return (int)ProjCfg<32>::kSmemBytes;
        case 256: return (int)ProjCfg<256>::kSmemBytes;
        default: return -1;
    }
}

cudaError_t proj_configure(int bn) {
    switch (bn) {
        case 16: return configure_bn<16>();
        case 32: return configure_bn<32>();
        case 256: return configure_bn<256>();
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t proj_launch(int bn, const CUtensorMap &map_h, const CUtensorMap &map_wl,
                        const CUtensorMap &map_wr, const ProjArgs &args, cudaStream_t stream) {
    switch (bn) {
        case 16: return launch_bn<16>(map_h, map_wl, map_wr, args, stream);
        case 32: return launch_bn<32>(map_h, map_wl, map_wr, args, stream);
        case 256: return launch_bn<256>(map_h, map_wl, map_wr, args, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace route
