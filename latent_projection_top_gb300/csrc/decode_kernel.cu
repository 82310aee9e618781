// Decode route step (1..20 token rows): steps a1..a4 in one kernel.
//
//   latent[r, n] = bf16( sum_k hidden[r, k] * W_latent[k, n] )   n < 3584
//   logits[r, e] =       sum_k hidden[r, k] * W_router[k, e]    e < 896
//   ids / weights = top-16 of logits[r, :]
//
// At decode widths the step is a stream of the 64.2 MB of weights; the
// arithmetic is small.  The kernel is built around that stream.
//
// Work split.  The weights are cut into 18 column tiles of 256 columns (14
// latent, 4 router; the last router tile has 128 real columns and TMA
// zero-fills the rest) and 112 k-blocks of 64.  The grid is 36 clusters of
// four CTAs, one CTA per SM (144 SMs); clusters 2t and 2t+1 cover tile t and
// each of their CTAs streams 14 consecutive k-blocks of it.  256-column tiles
// put 512 contiguous bytes per weight row in flight, which the HBM needs to
// run at full speed.
//
// Per CTA.  A TMA producer brings, per k-block, four 64x64 weight boxes and
// the hidden box (BN = 16 or 32 rows, zero-filled past `rows`) into a 6-stage
// shared-memory ring; one thread issues tcgen05 MMAs (128 weight columns on
// M, token rows on N) into a fresh TMEM accumulator per k-block; four
// epilogue warps add each k-block's FP32 result into a two-float (TwoSum)
// running sum, so the only rounding left is the tensor core's inside one
// 64-long block.
//
// Reduction, all in a fixed order (bitwise reproducible, and a row's bits do
// not depend on the number of rows):
//   1. the four CTAs of a cluster exchange their partials through distributed
//      shared memory; CTA j sums columns [64j, 64j+64) over ranks 0..3;
//   2. the two clusters of a tile meet in global scratch: the second to
//      arrive adds half 0 then half 1, rounds once and writes the outputs.
// Top-16: the 8 CTAs of the half-width router tile finish their stream first;
// once all 16 router column slices are final (a bounded wait on a counter
// that the slice writers raise), their warps run the top-16, one row each.
//
// Programmatic dependent launch: the kernel lets its successor launch at
// once and prefetches its first weight boxes (model parameters, which no
// predecessor writes) before `griddepcontrol.wait`; it reads the hidden rows
// and touches global scratch and outputs only after the wait.
//
// Every wait is bounded (timeout_ns): on expiry the kernel sets the status
// word, drains its in-flight copies and MMAs, frees TMEM and returns; the
// cluster barriers are still passed by every CTA.
#include <cuda_bf16.h>

#include "common.cuh"
#include "sm103_ptx.cuh"
#include "topk16.cuh"

namespace route {
namespace {

constexpr uint32_t kBoxBytes = 64 * 64 * 2;         // one 64-column x 64-k weight box
constexpr uint32_t kDAStageBytes = 4 * kBoxBytes;   // 256 columns x 64 k
constexpr int kNumAcc = 8;                          // TMEM accumulator ring (k-blocks in flight)
constexpr int kWorkerCtas = 2 * kDClusterSize;      // CTAs of the last router tile run the top-16
constexpr int kTailThreads = kProjThreads;

template <int BN>
struct DecCfg {
    static constexpr uint32_t kBStageBytes = BN * 128;  // BN rows x 64 k, BF16
    static constexpr uint32_t kStageBytes = kDAStageBytes + kBStageBytes;
    static constexpr int kStages = 6;
    static constexpr uint32_t kAccCols = 2 * BN;       // two 128-column blocks per accumulator
    static constexpr uint32_t kTmemCols = kNumAcc * kAccCols <= 256 ? 256 : 512;
    static constexpr uint32_t kSmemBytes = 1024 + kStages * kStageBytes + 256;
    // tcgen05 kind::f16: FP32 accumulator, BF16 A (MN-major) and B (K-major),
    // N = BN token rows, M = 128 weight columns.
    static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) |
                                       ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    static_assert(BN == 16 || BN == 32, "decode row tile");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
    static_assert(kNumAcc * kAccCols <= kTmemCols, "TMEM");
    // the partial (rows x 256 two-floats) is staged in the freed stage ring
    static_assert(kDecodeMaxRows * kDTileCols * 8 <= kStages * kStageBytes, "partial staging");
};

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;  // descriptor version for tcgen05
    d |= 2ull << 61;  // 128-byte swizzle
    return d;
}

// Error-free addition (Knuth's TwoSum): hi + x = s + e exactly; e joins lo.
__device__ __forceinline__ void two_sum_acc(float &hi, float &lo, float x) {
    const float s = hi + x;
    const float bp = s - hi;
    const float e = (hi - (s - bp)) + (x - bp);
    hi = s;
    lo += e;
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
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

template <int BN>
__global__ void __launch_bounds__(kProjThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_wl,
                  const __grid_constant__ CUtensorMap map_wr, const __grid_constant__ DecodeArgs args) {
    using C = DecCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem_base;
    __shared__ volatile int s_abort;
    __shared__ unsigned s_pair, s_go;
    __shared__ uint2 s_cand[kProjThreads / 32][kCandMax];

    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    float2 *const stage_f2 = reinterpret_cast<float2 *>(smem_raw + (sbase - raw));
    const uint32_t bars = sbase + C::kStages * C::kStageBytes;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (C::kStages + s); };
    auto accfull_bar = [&](int b) { return bars + 8u * (2 * C::kStages + b); };
    auto accempty_bar = [&](int b) { return bars + 8u * (2 * C::kStages + kNumAcc + b); };
    const uint32_t drain_bar = bars + 8u * (2 * C::kStages + 2 * kNumAcc);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tid = threadIdx.x;
    const int cluster = blockIdx.x / kDClusterSize;
    const int rank = (int)ptx::cluster_ctarank();  // == blockIdx.x % 4
    const int t = cluster >> 1;                     // column tile
    const int half = cluster & 1;
    const int kb0 = (half * kDClusterSize + rank) * kDKPerCta;
    const bool lat = t < kDLatTiles;
    const int x0 = (lat ? t : t - kDLatTiles) * kDTileCols;
    const int rows = args.rows;

    if (tid == 0) {
        // Let the next kernel on the stream launch as soon as SMs free up.
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        s_abort = 0;
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < kNumAcc; ++b) {
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

    // epilogue state: the CTA's two-float partial for 2 columns x BN rows per thread
    float hi[2][BN], lo[2][BN];

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            const uint64_t pol_w = ptx::policy_evict_first();
            const uint64_t pol_h = ptx::policy_evict_last();
            const CUtensorMap *wmap = lat ? &map_wl : &map_wr;
            constexpr int n_pre = kDKPerCta < C::kStages ? kDKPerCta : C::kStages;
            auto weights_of = [&](int kb, uint32_t a, uint32_t bar) {
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    ptx::tma_load_2d(a + b * kBoxBytes, wmap, bar, x0 + 64 * b, kb * kKBlock, pol_w);
            };
            uint32_t armed = 0u, armed_par = 0u;
            // Weight boxes of the first stages go out before the grid
            // dependency resolves (no predecessor writes the weights).
            for (int i = 0; i < n_pre; ++i) {
                ptx::mbar_arrive_expect_tx(full_bar(i), C::kStageBytes);
                weights_of(kb0 + i, sbase + i * C::kStageBytes, full_bar(i));
                armed |= 1u << i;
            }
            asm volatile("griddepcontrol.wait;" ::: "memory");
            for (int i = 0; i < n_pre; ++i) {
                if (args.test_stall && i == kDKPerCta - 1) continue;  // test hook
                ptx::tma_load_2d(sbase + i * C::kStageBytes + kDAStageBytes, &map_h, full_bar(i),
                                 (kb0 + i) * kKBlock, 0, pol_h);
            }
            bool ok = true;
            for (int i = n_pre; i < kDKPerCta; ++i) {
                const int s = i % C::kStages;
                const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
                if (!wait_phase(empty_bar(s), ph ^ 1u, args, &s_abort)) {
                    ok = false;
                    break;
                }
                if (args.test_stall && i == kDKPerCta - 1) continue;  // test hook: never filled
                const uint32_t a = sbase + s * C::kStageBytes;
                ptx::mbar_arrive_expect_tx(full_bar(s), C::kStageBytes);
                weights_of(kb0 + i, a, full_bar(s));
                ptx::tma_load_2d(a + kDAStageBytes, &map_h, full_bar(s), (kb0 + i) * kKBlock, 0, pol_h);
                armed |= 1u << s;
                armed_par = (armed_par & ~(1u << s)) | (ph << s);
            }
            if (!ok || s_abort) {  // let every issued copy land before the stages are reused
                for (int s = 0; s < C::kStages; ++s)
                    if (armed & (1u << s)) wait_drain(full_bar(s), (armed_par >> s) & 1u, args);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer: one fresh accumulator per k-block ----------------
            for (int i = 0; i < kDKPerCta; ++i) {
                const int s = i % C::kStages;
                const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
                const int buf = i % kNumAcc;
                const uint32_t use = (uint32_t)(i / kNumAcc);
                if (!wait_phase(accempty_bar(buf), (use & 1u) ^ 1u, args, &s_abort)) break;
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
                        ptx::mma_bf16(d_tmem, da, db, C::kIdesc, kk > 0 ? 1u : 0u);
                    }
                }
                ptx::mma_commit(empty_bar(s));
                ptx::mma_commit(accfull_bar(buf));
            }
            ptx::mma_commit(drain_bar);  // every MMA retired before TMEM and smem are reused
            wait_drain(drain_bar, 0u, args);
        }
    } else {
        // ---------------- epilogue: two-float sums of the k-block results ----------------
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int r = 0; r < BN; ++r) hi[h][r] = lo[h][r] = 0.f;
        for (int i = 0; i < kDKPerCta; ++i) {
            const int buf = i % kNumAcc;
            const uint32_t use = (uint32_t)(i / kNumAcc);
            // Each warp waits on its own; an abort seen by one is seen by all.
            if (!wait_phase(accfull_bar(buf), use & 1u, args, &s_abort)) break;
            ptx::tc_fence_after();
            const uint32_t taddr =
                tmem_base + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(buf * C::kAccCols);
            uint32_t v[2][BN];
#pragma unroll
            for (int ch = 0; ch < BN / 16; ++ch) {
                ptx::tmem_ld_x16(taddr + ch * 16, *reinterpret_cast<uint32_t(*)[16]>(&v[0][ch * 16]));
                ptx::tmem_ld_x16(taddr + BN + ch * 16,
                                 *reinterpret_cast<uint32_t(*)[16]>(&v[1][ch * 16]));
            }
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(accempty_bar(buf));
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int r = 0; r < BN; ++r) two_sum_acc(hi[h][r], lo[h][r], __uint_as_float(v[h][r]));
        }
    }

    // ---------------- tail: every thread of every CTA passes here ----------------
    ptx::tc_fence_before();
    __syncthreads();  // MMAs retired, stage ring free, epilogue sums final
    if (warp >= 2) {
        // Stage this CTA's partial, [row][256 columns] two-floats, in the freed ring.
        const int col = 32 * (warp & 3) + lane;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int r = 0; r < BN; ++r)
                if (r < rows) stage_f2[r * kDTileCols + h * 128 + col] = make_float2(hi[h][r], lo[h][r]);
    }
    __syncthreads();
    ptx::cluster_sync();  // all four partials of the cluster are staged

    // 1. CTA `rank` sums columns [64 rank, 64 rank + 64) over ranks 0..3.
    constexpr int kMaxItems = (kDecodeMaxRows * kDSliceCols / 2 + kTailThreads - 1) / kTailThreads;
    float4 part[kMaxItems];  // (hi, lo) of two adjacent columns
    const int items = rows * (kDSliceCols / 2);
#pragma unroll
    for (int q = 0; q < kMaxItems; ++q) {
        const int it = tid + q * kTailThreads;
        if (it < items) {
            const int r = it / (kDSliceCols / 2);
            const int c = rank * kDSliceCols + 2 * (it % (kDSliceCols / 2));
            const uint32_t local = ptx::smem_addr(&stage_f2[r * kDTileCols + c]);
            float4 p[kDClusterSize];
#pragma unroll
            for (int k = 0; k < kDClusterSize; ++k) p[k] = ptx::ld_cluster_f4(ptx::map_to_rank(local, k));
            float h0 = 0.f, l0 = 0.f, h1 = 0.f, l1 = 0.f;
#pragma unroll
            for (int k = 0; k < kDClusterSize; ++k) {
                two_sum_acc(h0, l0, p[k].x);
                l0 += p[k].y;
                two_sum_acc(h1, l1, p[k].z);
                l1 += p[k].w;
            }
            part[q] = make_float4(h0, l0, h1, l1);
            // this cluster's half of the tile, for the other cluster to find
            float4 *dst = reinterpret_cast<float4 *>(
                args.ws + ((size_t)(t * 2 + half) * kDecodeMaxRows + r) * kDTileCols + c);
            *dst = part[q];
        }
    }
    __threadfence();      // publish this cluster's half before the arrival count below
    ptx::cluster_sync();  // peers' shared memory is no longer read

    // 2. The second of the tile's two clusters to arrive at slice `rank` finishes it.
    __syncthreads();
    if (tid == 0) s_pair = atomicAdd(&args.words[kWordPairs + t * kDClusterSize + rank], 1u);
    __syncthreads();
    const bool finisher = s_pair == 1u;
    if (finisher) {
        __threadfence();
#pragma unroll
        for (int q = 0; q < kMaxItems; ++q) {
            const int it = tid + q * kTailThreads;
            if (it < items) {
                const int r = it / (kDSliceCols / 2);
                const int c = rank * kDSliceCols + 2 * (it % (kDSliceCols / 2));
                const float4 other = __ldcg(reinterpret_cast<const float4 *>(
                    args.ws + ((size_t)(t * 2 + (1 - half)) * kDecodeMaxRows + r) * kDTileCols + c));
                const float4 a = half == 0 ? part[q] : other;  // fixed order: half 0, then half 1
                const float4 b = half == 0 ? other : part[q];
                float h0 = a.x, l0 = a.y, h1 = a.z, l1 = a.w;
                two_sum_acc(h0, l0, b.x);
                l0 += b.y;
                two_sum_acc(h1, l1, b.z);
                l1 += b.w;
                const float y0 = h0 + l0, y1 = h1 + l1;
                const int n = x0 + c;
                if (lat) {
                    *reinterpret_cast<uint32_t *>(args.latent + (size_t)r * kLatent + n) =
                        (uint32_t)bf16_bits(y0) | ((uint32_t)bf16_bits(y1) << 16);
                } else if (n < kExperts) {
                    *reinterpret_cast<float2 *>(args.logits + (size_t)r * kExperts + n) =
                        make_float2(y0, y1);
                }
            }
        }
        __syncthreads();
        if (tid == 0) {
            args.words[kWordPairs + t * kDClusterSize + rank] = 0u;  // ready for the next launch
            if (!lat) {
                __threadfence();
                const unsigned done = atomicAdd(&args.words[kWordRouterDone], 1u);
                if (!args.fuse_topk && done == kDRouterSlices - 1) args.words[kWordRouterDone] = 0u;
            }
        }
    }

    // 3. Top-16: the CTAs of the last (half-width) router tile, once every
    //    router slice is final.  Rows r = worker + 8 * warp.
    if (args.fuse_topk && t == kDTiles - 1) {
        const int worker = half * kDClusterSize + rank;
        if (tid == 0) {
            bool ok = !s_abort;
            const uint64_t t0 = ptx::global_timer_ns();
            while (ok && *(volatile unsigned *)&args.words[kWordRouterDone] < (unsigned)kDRouterSlices) {
                if (ptx::global_timer_ns() - t0 > args.timeout_ns) {
                    fail_timeout(args, &s_abort);
                    ok = false;
                }
            }
            __threadfence();
            s_go = ok ? 1u : 0u;
        }
        __syncthreads();
        if (s_go) {
            const int r = worker + kWorkerCtas * warp;
            if (r < rows)
                topk16_warp(args.logits + (size_t)r * kExperts, args.ids + (size_t)r * kTopK,
                            args.weights + (size_t)r * kTopK, lane, s_cand[warp]);
        }
        __syncthreads();
        if (tid == 0) {
            const unsigned w = atomicAdd(&args.words[kWordWorkersDone], 1u);
            if (w == kWorkerCtas - 1) {  // every worker is past its wait: reset for the next launch
                args.words[kWordRouterDone] = 0u;
                args.words[kWordWorkersDone] = 0u;
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

template <int BN>
cudaError_t configure_bn() {
    return cudaFuncSetAttribute(decode_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)DecCfg<BN>::kSmemBytes);
}

template <int BN>
cudaLaunchConfig_t launch_config(cudaStream_t stream, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t c = {};
    c.gridDim = dim3(kDGrid);
    c.blockDim = dim3(kProjThreads);
    c.dynamicSmemBytes = DecCfg<BN>::kSmemBytes;
    c.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kDClusterSize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    c.attrs = attr;
    c.numAttrs = 2;
    return c;
}

template <int BN>
cudaError_t max_clusters_bn(int *n) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t c = launch_config<BN>(nullptr, attr);
    c.numAttrs = 1;  // the cluster shape only
    return cudaOccupancyMaxActiveClusters(n, decode_kernel<BN>, &c);
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap &mh, const CUtensorMap &ml, const CUtensorMap &mr,
                      const DecodeArgs &a, cudaStream_t stream) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t c = launch_config<BN>(stream, attr);
    return cudaLaunchKernelEx(&c, decode_kernel<BN>, mh, ml, mr, a);
}

}  // namespace

int decode_bn_for(int rows) { return rows <= 16 ? 16 : 32; }

int decode_smem_bytes(int bn) {
    return bn == 16 ? (int)DecCfg<16>::kSmemBytes : bn == 32 ? (int)DecCfg<32>::kSmemBytes : -1;
}

cudaError_t decode_configure(int bn) {
    return bn == 16 ? configure_bn<16>() : bn == 32 ? configure_bn<32>() : cudaErrorInvalidValue;
}

cudaError_t decode_max_clusters(int bn, int *clusters) {
    return bn == 16 ? max_clusters_bn<16>(clusters)
           : bn == 32 ? max_clusters_bn<32>(clusters)
                      : cudaErrorInvalidValue;
}

cudaError_t decode_launch(int bn, const CUtensorMap &map_h, const CUtensorMap &map_wl,
                          const CUtensorMap &map_wr, const DecodeArgs &args, cudaStream_t stream) {
    return bn == 16   ? launch_bn<16>(map_h, map_wl, map_wr, args, stream)
           : bn == 32 ? launch_bn<32>(map_h, map_wl, map_wr, args, stream)
                      : cudaErrorInvalidValue;
}

}  // namespace route
