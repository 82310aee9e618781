// Shapes, launch arguments and internal launch entry points shared by the
// route library's translation units (kernels and the C ABI layer).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace route {

// Fixed route-step dimensions: K = 7168 hidden, 3584 latent columns
// ("Optionally gather the Kimi3 prefill latent instead of reducing it",
// Description, Compile bullet) and 896 = 56 x 16 experts ("Use two row
// blocks for eight-row Kimi paired gathers", body).
constexpr int kHidden = 7168;
constexpr int kLatent = 3584;
constexpr int kExperts = 896;
constexpr int kTopK = 16;
constexpr int kDecodeMaxRows = 20;

// K is consumed 64 at a time.
constexpr int kKBlock = 64;
constexpr int kKBlocks = kHidden / kKBlock;                 // 112
constexpr int kKSplitSlices = 8;                            // the general path's K slices (896 deep)
static_assert(kKBlocks % kKSplitSlices == 0, "K slices of whole k-blocks");
// Prefill tiling: one tile = 256 weight columns (the MMA M side, split over a
// pair of CTAs) x 256 token rows (the MMA N side; each CTA of the pair loads
// 128 of them): 14 latent + 4 router column tiles, the last with 128 real
// columns.
constexpr int kPrefillBN = 256;
constexpr int kPrefillColTiles = 18;
constexpr int kPrefillLatTiles = 14;
constexpr int kPrefillHiddenBoxRows = 64;
constexpr int kProjThreads = 320;                           // 10 warps

enum Mode : int { kDecode = 0, kPrefill = 1 };

// Device status bits (the kernels set them instead of hanging).
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusBounds = 2u;  // debug library: an index out of range was skipped

// ROUTE_IN_BOUNDS(ok, status): in the debug library (built with -DROUTE_DEBUG)
// every computed global index is checked before its access; a failed check
// sets kStatusBounds in the status word and the access is skipped, so the
// kernel neither faults nor traps.  In the release library it is `true`.
#ifdef ROUTE_DEBUG
__device__ __forceinline__ bool route_in_bounds(bool ok, unsigned *status) {
    if (!ok) atomicOr(status, kStatusBounds);
    return ok;
}
#define ROUTE_IN_BOUNDS(ok, status) route_in_bounds((ok), (status))
#else
#define ROUTE_IN_BOUNDS(ok, status) true
#endif

// Prefill work is a list of tiles per CTA pair, built on the host.  A tile
// is 256 weight columns (one column tile c: 0..13 latent, 14..17 router) by
// the 256 token rows from row0 on, computed as one FP32 accumulation over
// the whole K, or (K-split kind, latent tiles) as eight 896-deep K slices
// whose results are rounded to BF16 and added in FP32 (the general path's
// latent).  Packed into one int: row0 (a multiple of 256) + 32 * kind + c.
enum PrefillTileKind : int { kTileFull = 0, kTileKsplit = 1 };
__host__ __device__ constexpr int pack_tile(int c, int kind, int row0) { return row0 + 32 * kind + c; }
__host__ __device__ constexpr int tile_col(int t) { return t & 31; }
__host__ __device__ constexpr int tile_kind(int t) { return (t >> 5) & 3; }
__host__ __device__ constexpr int tile_row0(int t) { return t & ~255; }

// Longest tile list of one pair (the host checks it): 65536 rows give 4608
// tiles over 76 pairs, at most 61 a pair.
constexpr int kMaxPairTiles = 256;

// Per-row latent sum-of-squares parts written by the prefill epilogue: one
// per (latent column tile, CTA of the pair, 32-column warp group).
constexpr int kSsParts = kPrefillLatTiles * 2 * 4;          // 112

// Everything the prefill projection kernel needs besides its tensor maps.
struct ProjArgs {
    int rows;            // token rows in this call
    int grid;            // persistent CTAs launched (pairs of CTAs: even)
    int test_stall;      // test hook: skip each CTA's last copy so a wait must time out
    int overlap;         // read hidden before the grid dependency resolves
    unsigned long long timeout_ns;  // bound on every wait inside the kernel
    unsigned *status;          // device status word
    const int *sched;          // packed tiles of every pair, pair after pair
    const int *sched_off;      // pair p's tiles: sched[sched_off[p] .. sched_off[p + 1])
    float2 *ss_part;           // optional [rows][kSsParts] latent sum-of-squares parts (hi, lo)
    int n_latent;              // latent columns stored: 3584, or a column shard's share
    int n_experts;             // router columns of W_router: 896, or a column shard's share
};

// Decode split-K: 18 column tiles of 256 columns (14 latent, 4 router -- the
// last router tile holds 128 real columns) x 112 k-blocks.
constexpr int kDTileCols = 256;
constexpr int kDLatTiles = kLatent / kDTileCols;                           // 14
constexpr int kDRouterTiles = (kExperts + kDTileCols - 1) / kDTileCols;    // 4
constexpr int kDTiles = kDLatTiles + kDRouterTiles;                        // 18
constexpr int kMaxGrid = 256;
// device words: [0] status (the rest spare)
constexpr int kWordStatus = 0;
constexpr int kWords = 64;

struct DecodeArgs {
    int rows;            // 1..20
    int grid;            // CTAs of the stream kernel (<= kMaxGrid)
    int test_stall;      // test hook: skip each CTA's last copy so a wait must time out
    int overlap;         // read hidden before the grid dependency resolves
    int ksplit;          // latent with the general path's K-split arithmetic
    int lat_tiles;       // latent column tiles (14; a column shard's: ceil(its columns / 256))
    int tiles;           // latent + router column tiles (18, or a column shard's)
    int pre_l2;          // units after the first ring whose weights go to L2 at the CTA's start
    unsigned long long timeout_ns;
    int cta_unit[kMaxGrid + 1];  // CTA g owns units [cta_unit[g], cta_unit[g+1]); unit u =
                                 // (tile u / 112, k-block u % 112)
    int seg_base[kDTiles];       // first partial slot of tile t
    int seg_count[kDTiles];      // CTAs (partials) covering tile t
    int cta_first[kDTiles];      // first CTA covering tile t
    float2 *ws;                  // partials [slot][kDecodeMaxRows][256] as (hi, lo)
    unsigned *words;             // device status word
    uint16_t *latent;
    float *logits;
    int32_t *ids;
    float *weights;
    float *sumsq;                // optional [rows]: sum of squares of each latent row
    // With overlap set, hidden rows published by a concurrent staging kernel:
    // the stream kernel reads them once *hidden_count >= hidden_target
    // (acquire; null: no wait).
    const unsigned *hidden_count = nullptr;
    unsigned hidden_target = 0;
};

// Internal launchers (defined next to their kernels).  Every launch uses
// programmatic dependent launch (see the kernels for what each waits on).
int prefill_smem_bytes();
cudaError_t prefill_configure();
// map_lat / map_lg: store maps of the latent [rows, 3584] BF16 and the logits
// [rows, 896] FP32 with 32-column x 16-row boxes.
cudaError_t prefill_launch(const CUtensorMap &map_h, const CUtensorMap &map_wl,
                           const CUtensorMap &map_wr, const CUtensorMap &map_lat,
                           const CUtensorMap &map_lg, const ProjArgs &args, cudaStream_t stream);

int decode_bn_for(int rows);
int decode_smem_bytes(int bn);
cudaError_t decode_configure(int bn);
cudaError_t decode_launch(int bn, const CUtensorMap &map_h, const CUtensorMap &map_wl,
                          const CUtensorMap &map_wr, const DecodeArgs &args, int do_topk,
                          cudaStream_t stream);

// Copy `bytes` (a multiple of 16) from page-locked host memory, through its
// device-mapped address, into device memory; PDL-chained like the route
// kernels.
cudaError_t stage_in_launch(const void *src_mapped, void *dst, size_t bytes, cudaStream_t stream);
cudaError_t host_done_launch(unsigned *counter, unsigned *flag_mapped, cudaStream_t stream);
// The same copy for a step whose stream kernel does not wait for it to
// complete: it writes `dst` once *done_counter >= need (the buffer's last
// reader has finished), then adds one per CTA to *published (release) and,
// last, waits for its own predecessor.  *ctas receives the CTAs launched.
cudaError_t stage_publish_launch(const void *src_mapped, void *dst, size_t bytes,
                                 const unsigned *done_counter, unsigned need, unsigned *published,
                                 unsigned *status, unsigned long long timeout_ns, int *ctas,
                                 cudaStream_t stream);

// The top-16 of each row; with `sumsq` non-null also the row's latent sum
// of squares (the sum of its kSsParts parts in `ss_part`, which the same
// predecessor wrote).
cudaError_t topk_launch(const float *logits, int rows, int32_t *ids, float *weights,
                        const float2 *ss_part, float *sumsq, cudaStream_t stream);

// A column shard at decode sizes (1..20 rows): the split-K weight stream over
// the shard's args.tiles column tiles, then a kernel that sums the partials
// into the shard's latent [rows, n_lat] and logits [rows, n_exp] (args.latent,
// args.logits) and writes the shard's top-16 as candidates (global ids
// id_base + local id, and their logits).
cudaError_t decode_shard_launch(int bn, const CUtensorMap &map_h, const CUtensorMap &map_wl,
                                const CUtensorMap &map_wr, const DecodeArgs &args, int n_lat,
                                int n_exp, int id_base, int32_t *cand_ids, float *cand_logits,
                                cudaStream_t stream);

// A column shard's local top-16: of the `n` logits of each row (row stride
// n), the 16 largest (the same ranking), written as global expert ids
// (id_base + local id) and their logits.
cudaError_t shard_topk_launch(const float *logits, int rows, int n, int id_base, int32_t *cand_ids,
                              float *cand_logits, cudaStream_t stream);

// The top-16 of each row over num_shards x 16 candidates (shard-major:
// [shard][row][16] ids and logits) and their routing weights.
cudaError_t merge_launch(const int32_t *cand_ids, const float *cand_logits, int rows,
                         int num_shards, int32_t *ids, float *weights, cudaStream_t stream);

// Column shards: shard s of W owns latent columns [kLatent s / W, kLatent
// (s+1) / W) and experts [kExperts s / W, kExperts (s+1) / W).
constexpr int kMaxShards = 16;

}  // namespace route
