// C ABI of the route library: plan preparation (envelope checks, launch
// geometry, split-K partition, scratch), argument validation and launches.
// Every check happens on the host before anything is enqueued; failures are
// status codes plus a per-thread message.
#include <cuda.h>
#include <cuda_runtime.h>

#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "common.cuh"
#include "route.h"

using namespace route;

struct route_plan {
    int mode;
    int rows;
    int device;
    int bn;                   // decode: 16 or 32 token rows per MMA; prefill: 256
    int grid;
    int segments;
    ProjArgs pre;             // prefill launch arguments (per-call pointers added at launch)
    DecodeArgs dec;           // decode launch arguments, incl. the split-K partition
    float2 *ws;               // decode: split-K partials, then the sum-of-squares parts;
                              // prefill: the per-row latent sum-of-squares parts
    size_t ws_bytes;          // both
    int *sched;               // prefill: the pairs' tile lists (device), plain and K-split
    const int *sched_tiles[2], *sched_off[2];  // [0] plain, [1] K-split latent
    int sched_pairs[2];
    int pre_ksplit;           // prefill: latent with the general path's K-split arithmetic
    int num_shards;           // column-shard plans: W (0 for a plan of the whole layer)
    int shard;                // column-shard plans: this plan's shard, 0 .. W-1
    int n_lat, n_exp;         // latent columns and experts the plan computes
    unsigned *words;          // device status word (+ spare)
    uint8_t *staging;         // device staging for route_step_host
    size_t staging_bytes;
    // The last tensor map made for each operand (a map describes an address
    // and a shape; the shapes are fixed per plan, so an equal address reuses
    // it and skips the encode on the next call).
    struct MapCache {
        const void *ptr = nullptr;
        CUtensorMap map;
    };
    mutable MapCache map_h, map_wl, map_wr, map_lat, map_lg;
    route_host_step *steps = nullptr;  // prepared host steps, released with the plan
};

// A captured route_step_host (decode, page-locked buffers): staging kernel,
// stream kernel, finish kernel.
struct route_host_step {
    route_plan *plan;         // NULL once the plan is gone
    route_host_step *next;    // the plan's list
    cudaGraph_t graph;
    cudaGraphExec_t exec;
    cudaStream_t stream;      // the caller's stream: launches there
    // Completion: the graph's last kernel stores the step's number into a
    // page-locked word (flag_host; flag_dev is its mapped address) after a
    // system-scope fence; run() waits for that number instead of for the
    // stream.  counter is the device copy of the number.
    unsigned *flag_host;
    unsigned *flag_dev;
    unsigned *counter;
    unsigned launched;        // the number of the last step launched
    unsigned done;            // the number of the last step seen complete
    // For direct launches (route_host_step_launch): the mapped hidden rows,
    // the weights, and the plan's decode arguments as they were at creation
    // with this step's outputs filled in -- what the graph holds.
    const void *hidden_mapped, *W_latent, *W_router;
    route::DecodeArgs dec;
    // Direct launches stage the hidden rows into two buffers of the step's
    // own, alternately (hbuf, hbuf + hbuf_stride; hmap: their tensor maps),
    // and publish them through the device word `published` (one addition
    // per staging CTA; published_total: the sum after the last launch).
    // buf_launch[j]: the number of the launch that last read buffer j.
    uint8_t *hbuf;
    size_t hbuf_stride;
    CUtensorMap hmap[2];
    unsigned *published;
    unsigned published_total;
    unsigned staged;
    unsigned buf_launch[2];
};

namespace {

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // bound on every in-kernel wait
constexpr long long kHostWaitNs = 4000000000ll;  // a host step's wait for its completion word

thread_local char g_err[512] = "";

route_status fail(route_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

route_status cuda_fail(cudaError_t e, const char *what) {
    return fail(ROUTE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_encode_mu;
EncodeTiledFn g_encode = nullptr;

route_status get_encode(EncodeTiledFn *out) {
    std::lock_guard<std::mutex> lk(g_encode_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
            return fail(ROUTE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    *out = g_encode;
    return ROUTE_OK;
}

// 2-D row-major tensor map (zero fill out of bounds): BF16 operands with
// 128-byte swizzle for the MMA loads; for the prefill stores, BF16 or FP32
// without swizzle.
route_status encode_2d(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer,
                       uint32_t box_inner, uint32_t box_outer, const char *what,
                       bool fp32 = false, bool swizzle = true) {
    EncodeTiledFn enc = nullptr;
    route_status st = get_encode(&enc);
    if (st != ROUTE_OK) return st;
    const uint64_t esize = fp32 ? 4 : 2;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * esize};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ROUTE_ERR_CUDA, "tensor map for %s rejected (CUresult %d)", what, (int)r);
    return ROUTE_OK;
}

struct DeviceGuard {
    int prev = -1;
    bool changed = false;
    cudaError_t err = cudaSuccess;
    explicit DeviceGuard(int dev) {
        err = cudaGetDevice(&prev);
        if (err == cudaSuccess && prev != dev) {
            err = cudaSetDevice(dev);
            changed = (err == cudaSuccess);
        }
    }
    ~DeviceGuard() {
        if (changed) cudaSetDevice(prev);
    }
};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

void release_step_graph(route_host_step *h) {
    if (h->exec) cudaGraphExecDestroy(h->exec);
    if (h->graph) cudaGraphDestroy(h->graph);
    if (h->counter) cudaFree(h->counter);
    if (h->flag_host) cudaFreeHost(h->flag_host);
    if (h->hbuf) cudaFree(h->hbuf);
    h->exec = nullptr;
    h->graph = nullptr;
    h->counter = nullptr;
    h->flag_host = h->flag_dev = nullptr;
    h->hbuf = nullptr;
    h->published = nullptr;
}

void free_plan(route_plan *p) {
    if (!p) return;
    for (route_host_step *h = p->steps; h; h = h->next) {  // the steps outlive it, inert
        release_step_graph(h);
        h->plan = nullptr;
    }
    if (p->ws) cudaFree(p->ws);
    if (p->sched) cudaFree(p->sched);
    if (p->words) cudaFree(p->words);
    if (p->staging) cudaFree(p->staging);
    delete p;
}

// Staging layout for route_step_host: hidden, latent, logits, ids, weights.
struct Staging {
    void *hidden, *latent;
    float *logits, *weights;
    int32_t *ids;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

Staging staging_of(const route_plan *p) {
    size_t r = (size_t)p->rows;
    uint8_t *b = p->staging;
    Staging s;
    s.hidden = b;
    b += align256(r * kHidden * 2);
    s.latent = b;
    b += align256(r * kLatent * 2);
    s.logits = reinterpret_cast<float *>(b);
    b += align256(r * kExperts * 4);
    s.ids = reinterpret_cast<int32_t *>(b);
    b += align256(r * kTopK * 4);
    s.weights = reinterpret_cast<float *>(b);
    return s;
}

size_t staging_size(int rows) {
    size_t r = (size_t)rows;
    return align256(r * kHidden * 2) + align256(r * kLatent * 2) + align256(r * kExperts * 4) +
           align256(r * kTopK * 4) + align256(r * kTopK * 4);
}

route_status check_plan(const route_plan *p) {
    if (!p) return fail(ROUTE_ERR_NULL, "plan is NULL");
    return ROUTE_OK;
}

route_status cached_map(route_plan::MapCache &c, const void *ptr, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer, const char *what, CUtensorMap *out,
                        bool fp32 = false, bool swizzle = true) {
    if (c.ptr != ptr) {
        route_status st = encode_2d(&c.map, ptr, inner, outer, box_inner, box_outer, what, fp32,
                                    swizzle);
        if (st != ROUTE_OK) {
            c.ptr = nullptr;
            return st;
        }
        c.ptr = ptr;
    }
    *out = c.map;
    return ROUTE_OK;
}

route_status encode_all(const route_plan *p, const void *hidden, const void *W_latent,
                        const void *W_router, CUtensorMap *mh, CUtensorMap *ml, CUtensorMap *mr) {
    route_status st;
    // decode: one box holds the step's rows; prefill: each CTA of a pair
    // loads half of a tile's token rows
    const uint32_t hbox = p->mode == ROUTE_DECODE ? (uint32_t)p->bn : (uint32_t)kPrefillHiddenBoxRows;
    if ((st = cached_map(p->map_h, hidden, kHidden, (uint64_t)p->rows, kKBlock, hbox, "hidden",
                         mh)) != ROUTE_OK)
        return st;
    if ((st = cached_map(p->map_wl, W_latent, (uint64_t)p->n_lat, kHidden, 64, kKBlock, "W_latent",
                         ml)) != ROUTE_OK)
        return st;
    return cached_map(p->map_wr, W_router, (uint64_t)p->n_exp, kHidden, 64, kKBlock, "W_router", mr);
}

// The projection (and, for decode with do_topk, the top-16) of one step.
route_status launch_forward(const route_plan *p, const void *hidden, const void *W_latent,
                            const void *W_router, void *latent, float *logits, int32_t *ids,
                            float *weights, int do_topk, float *sumsq, cudaStream_t stream,
                            bool after_copy_in = false) {
    CUtensorMap mh, ml, mr;
    route_status st = encode_all(p, hidden, W_latent, W_router, &mh, &ml, &mr);
    if (st != ROUTE_OK) return st;
    cudaError_t e;
    if (p->mode == ROUTE_DECODE) {
        DecodeArgs a = p->dec;
        a.latent = static_cast<uint16_t *>(latent);
        a.logits = logits;
        a.ids = ids;
        a.weights = weights;
        a.sumsq = sumsq;
        // After the host path's copy in (a staging kernel or a copy), hidden
        // is the predecessor's output.
        if (after_copy_in) a.overlap = 0;
        e = decode_launch(p->bn, mh, ml, mr, a, do_topk, stream);
        if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
    } else {
        // the epilogue's TMA stores: 32 columns x 16 rows per box
        CUtensorMap mlat, mlg;
        if ((st = cached_map(p->map_lat, latent, (uint64_t)p->n_lat, (uint64_t)p->rows, 32, 16,
                             "latent", &mlat, false, false)) != ROUTE_OK ||
            (st = cached_map(p->map_lg, logits, (uint64_t)p->n_exp, (uint64_t)p->rows, 32, 16,
                             "logits", &mlg, true, false)) != ROUTE_OK)
            return st;
        ProjArgs a = p->pre;
        const int ks = p->pre_ksplit ? 1 : 0;
        a.sched = p->sched_tiles[ks];
        a.sched_off = p->sched_off[ks];
        a.grid = 2 * p->sched_pairs[ks];
        a.ss_part = sumsq != nullptr ? p->ws : nullptr;
        if (after_copy_in) a.overlap = 0;
        e = prefill_launch(mh, ml, mr, mlat, mlg, a, stream);
        if (e != cudaSuccess) return cuda_fail(e, "prefill kernel launch");
        if (do_topk) {
            e = topk_launch(logits, p->rows, ids, weights, p->ws, sumsq, stream);
            if (e != cudaSuccess) return cuda_fail(e, "top-16 kernel launch");
        }
    }
    return ROUTE_OK;
}

route_status check_whole_plan(const route_plan *p) {
    route_status st = check_plan(p);
    if (st != ROUTE_OK) return st;
    if (p->num_shards != 0)
        return fail(ROUTE_ERR_PLAN, "a column-shard plan runs route_shard_step only");
    return ROUTE_OK;
}

route_status check_forward_args(const route_plan *p, const void *hidden, const void *W_latent,
                                const void *W_router, const void *latent, const float *logits) {
    route_status st = check_whole_plan(p);
    if (st != ROUTE_OK) return st;
    if (!hidden || !W_latent || !W_router || !latent || !logits)
        return fail(ROUTE_ERR_NULL, "hidden, W_latent, W_router, latent and logits must be non-NULL");
    if (!aligned16(hidden) || !aligned16(W_latent) || !aligned16(W_router) || !aligned16(latent) ||
        !aligned16(logits))
        return fail(ROUTE_ERR_ALIGN, "every device pointer must be 16-byte aligned");
    return ROUTE_OK;
}

route_status check_topk_args(const route_plan *p, const float *logits, const int32_t *ids,
                             const float *weights) {
    route_status st = check_whole_plan(p);
    if (st != ROUTE_OK) return st;
    if (!logits || !ids || !weights)
        return fail(ROUTE_ERR_NULL, "logits, ids and weights must be non-NULL");
    if (!aligned16(logits) || !aligned16(ids) || !aligned16(weights))
        return fail(ROUTE_ERR_ALIGN, "every device pointer must be 16-byte aligned");
    return ROUTE_OK;
}

route_status run_step(const route_plan *p, const void *hidden, const void *W_latent,
                      const void *W_router, void *latent, float *logits, int32_t *ids,
                      float *weights, cudaStream_t stream, float *sumsq = nullptr) {
    return launch_forward(p, hidden, W_latent, W_router, latent, logits, ids, weights, 1, sumsq,
                          stream);
}

// Prefill work lists.  The tiles of a call, in column bands: a band of B
// column tiles over every 256-row block, then the next band, with B = the
// pair count over the row blocks (at least 1, at most all the columns), so
// that the pairs at work at one time read few weight tiles and every hidden
// row block.  Each tile goes, in that order, to the pair with the fewest
// tiles so far.  The column tiles are the first `lat_tiles` latent tiles and
// the first `router_tiles` router tiles (all 14 and 4 for a whole layer).
bool build_schedule(int rows, bool ksplit, int max_pairs, int lat_tiles, int router_tiles,
                    std::vector<int> &off, std::vector<int> &tiles, int *pairs) {
    std::vector<int> cols;
    for (int c = 0; c < lat_tiles; ++c) cols.push_back(c);
    for (int c = 0; c < router_tiles; ++c) cols.push_back(kPrefillLatTiles + c);
    const int ncols = (int)cols.size();
    const int row_blocks = (rows + kPrefillBN - 1) / kPrefillBN;
    int band = max_pairs / row_blocks;
    band = band < 1 ? 1 : band > ncols ? ncols : band;
    std::vector<int> order;
    for (int c0 = 0; c0 < ncols; c0 += band)
        for (int r = 0; r < row_blocks; ++r)
            for (int ci = c0; ci < c0 + band && ci < ncols; ++ci) {
                const int c = cols[ci], row0 = r * kPrefillBN;
                order.push_back(
                    pack_tile(c, ksplit && c < kPrefillLatTiles ? kTileKsplit : kTileFull, row0));
            }
    const int np = max_pairs < (int)order.size() ? max_pairs : (int)order.size();
    std::vector<std::vector<int>> lists(np);
    std::vector<int> load(np, 0);
    for (int t : order) {
        int best = 0;
        for (int q = 1; q < np; ++q)
            if (load[q] < load[best]) best = q;
        lists[best].push_back(t);
        load[best] += 1;
    }
    off.assign(1, 0);
    tiles.clear();
    for (auto &l : lists) {
        if ((int)l.size() > kMaxPairTiles) return false;
        tiles.insert(tiles.end(), l.begin(), l.end());
        off.push_back((int)tiles.size());
    }
    *pairs = np;
    return true;
}

// Decode stream grid: the largest CTA count, at most one per SM and at most
// `cap`, that divides the tiles * 112 (tile, k-block) units into equal, even
// runs: every CTA streams the same number of bytes, and its k-blocks pair up
// on one accumulator without a pair crossing a tile (tiles start at even
// units).  The whole layer's 18 tiles: 144 CTAs of 14 units on 152 SMs.
// At most 64 CTAs a tile: a column shard's finish sums a value's partials
// with up to four threads of at most 16 each, one memory round trip (this
// binds only a column shard's few tiles).  Never below the tile count, which
// route_prepare requires of the device.
int decode_grid(int sms, int cap, int tiles = kDTiles) {
    const int U = tiles * kKBlocks;
    int hi = sms < cap ? sms : cap;
    hi = hi < 64 * tiles ? hi : 64 * tiles;
    for (int g = hi; g > tiles; --g)
        if ((U / 2) % g == 0) return g;
    return tiles;
}

// Units past the first ring whose weights a decode CTA sends to L2 at its
// start.  Measured, interleaved in one process: 2 takes 0.24-0.45 us off a
// layer at 1-16 rows and 0.10-0.18 us at 20 rows with overlap, 0.06-0.42 us
// without, 0.25 us after a producer kernel; 3 and more are slower at 16-20
// rows.
constexpr int kDecodePreL2 = 2;

// Decode split-K partition: CTA g owns a contiguous run of (tile, k-block)
// units, the same number (+-1) for every CTA.
void decode_partition(DecodeArgs &a, int grid, int *segments, int lat_tiles = kDLatTiles,
                      int tiles = kDTiles) {
    const int U = tiles * kKBlocks;
    a.grid = grid;
    a.lat_tiles = lat_tiles;
    a.pre_l2 = kDecodePreL2;
    a.tiles = tiles;
    for (int g = 0; g <= grid; ++g) a.cta_unit[g] = (int)((long long)U * g / grid);
    int slots = 0;
    for (int t = 0; t < tiles; ++t) {
        const int first_u = t * kKBlocks, last_u = first_u + kKBlocks - 1;
        int g_first = -1, g_last = -1;
        for (int g = 0; g < grid; ++g) {
            if (a.cta_unit[g] <= first_u && first_u < a.cta_unit[g + 1]) g_first = g;
            if (a.cta_unit[g] <= last_u && last_u < a.cta_unit[g + 1]) g_last = g;
        }
        a.cta_first[t] = g_first;
        a.seg_count[t] = g_last - g_first + 1;
        a.seg_base[t] = slots;
        slots += a.seg_count[t];
    }
    *segments = slots;
}

// ---- allocation-free decode step ---------------------------------------
//
// route_step_decode_noalloc keeps its split-K scratch in this file-scope
// device array instead of memory from cudaMalloc.  Layout: a 256-byte word
// area (the kernels' status word) followed by the partial slots
// [slot][20 rows][256 columns] of (hi, lo) floats.  The slot count bounds the
// grid: a CTA's run spans at most two column tiles, so grid G needs at most
// G + 17 slots; the grid is capped at kNoAllocMaxGrid CTAs.
constexpr int kNoAllocMaxGrid = 160;
constexpr int kNoAllocMaxSlots = kNoAllocMaxGrid + kDTiles - 1;  // 177
constexpr size_t kNoAllocWordBytes = 256;
constexpr size_t kNoAllocSlotBytes = (size_t)kDecodeMaxRows * kDTileCols * sizeof(float2);
constexpr size_t kNoAllocScratchBytes = kNoAllocWordBytes + kNoAllocMaxSlots * kNoAllocSlotBytes;
static_assert(kWords * sizeof(unsigned) <= kNoAllocWordBytes, "word area");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Per-device set-up, done on the first call with that device current: the
// device address of g_noalloc_scratch (host code may not use the symbol
// itself), the kernels' shared-memory opt-in and the split-K partition.
struct NoAllocDevice {
    bool ready = false;
    unsigned char *scratch = nullptr;
    DecodeArgs base;
};
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc[kNoAllocMaxDevices];

route_status noalloc_setup(int device, NoAllocDevice **out) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    NoAllocDevice &d = g_noalloc[device];
    if (d.ready) {
        *out = &d;
        return ROUTE_OK;
    }
    cudaDeviceProp prop;
    cudaError_t e = cudaGetDeviceProperties(&prop, device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
    if (prop.major != 10 || prop.minor != 3)
        return fail(ROUTE_ERR_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a only",
                    device, prop.major, prop.minor);
    if (prop.multiProcessorCount < kDTiles)
        return fail(ROUTE_ERR_DEVICE, "decode needs at least %d SMs; device has %d", kDTiles,
                    prop.multiProcessorCount);
    for (int bn : {16, 32}) {
        if ((size_t)decode_smem_bytes(bn) > prop.sharedMemPerBlockOptin)
            return fail(ROUTE_ERR_DEVICE, "decode kernel needs %d B of shared memory per block",
                        decode_smem_bytes(bn));
        if ((e = decode_configure(bn)) != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    }
    EncodeTiledFn enc = nullptr;
    route_status st = get_encode(&enc);
    if (st != ROUTE_OK) return st;
    void *ptr = nullptr;
    if ((e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch)) != cudaSuccess)
        return cuda_fail(e, "cudaGetSymbolAddress(no-allocation scratch)");
    memset(&d.base, 0, sizeof d.base);
    const int grid = decode_grid(prop.multiProcessorCount, kNoAllocMaxGrid);
    int slots = 0;
    decode_partition(d.base, grid, &slots);
    if (slots > kNoAllocMaxSlots)
        return fail(ROUTE_ERR_PLAN, "partition needs %d scratch slots; the array holds %d", slots,
                    kNoAllocMaxSlots);
    d.scratch = static_cast<unsigned char *>(ptr);
    d.base.timeout_ns = kDefaultTimeoutNs;
    d.base.words = reinterpret_cast<unsigned *>(d.scratch);
    d.base.ws = reinterpret_cast<float2 *>(d.scratch + kNoAllocWordBytes);
    d.ready = true;
    *out = &d;
    return ROUTE_OK;
}

// A plan of the whole layer (num_shards == 0) or of column shard `shard` of
// `num_shards` (prefill kernel; checked by the caller).
route_status prepare_plan(int mode, int rows, int device, int shard, int num_shards,
                          route_plan **out) {
    g_err[0] = '\0';
    if (!out) return fail(ROUTE_ERR_NULL, "out is NULL");
    *out = nullptr;
    if (mode != ROUTE_DECODE && mode != ROUTE_PREFILL)
        return fail(ROUTE_ERR_MODE, "mode %d is neither ROUTE_DECODE (0) nor ROUTE_PREFILL (1)", mode);
    if (mode == ROUTE_DECODE && (rows < 1 || rows > ROUTE_DECODE_MAX_ROWS))
        return fail(ROUTE_ERR_ROWS, "decode prepares 1-%d rows; got %d", ROUTE_DECODE_MAX_ROWS, rows);
    if (mode == ROUTE_PREFILL && (rows < 1 || rows > ROUTE_PREFILL_MAX_ROWS))
        return fail(ROUTE_ERR_ROWS, "prefill prepares 1-%d rows; got %d", ROUTE_PREFILL_MAX_ROWS, rows);

    int ndev = 0;
    cudaError_t e = cudaGetDeviceCount(&ndev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
    if (device < 0 || device >= ndev)
        return fail(ROUTE_ERR_DEVICE, "device %d does not exist (%d devices)", device, ndev);
    cudaDeviceProp prop;
    if ((e = cudaGetDeviceProperties(&prop, device)) != cudaSuccess)
        return cuda_fail(e, "cudaGetDeviceProperties");
    if (prop.major != 10 || prop.minor != 3)
        return fail(ROUTE_ERR_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a only",
                    device, prop.major, prop.minor);
    EncodeTiledFn enc = nullptr;
    route_status st = get_encode(&enc);
    if (st != ROUTE_OK) return st;

    DeviceGuard guard(device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");

    route_plan *p = new (std::nothrow) route_plan();
    if (!p) return fail(ROUTE_ERR_PLAN, "out of host memory");
    p->mode = mode;
    p->rows = rows;
    p->device = device;
    p->num_shards = num_shards;
    p->shard = shard;
    p->n_lat = num_shards ? kLatent / num_shards : kLatent;
    p->n_exp = num_shards ? kExperts / num_shards : kExperts;
    p->bn = mode == ROUTE_DECODE ? decode_bn_for(rows) : kPrefillBN;
    const int smem = mode == ROUTE_DECODE ? decode_smem_bytes(p->bn) : prefill_smem_bytes();
    if (smem < 0 || (size_t)smem > prop.sharedMemPerBlockOptin) {
        free_plan(p);
        return fail(ROUTE_ERR_DEVICE, "kernel needs %d B of shared memory per block; device allows %zu",
                    smem, (size_t)prop.sharedMemPerBlockOptin);
    }
    if ((e = mode == ROUTE_DECODE ? decode_configure(p->bn) : prefill_configure()) != cudaSuccess) {
        free_plan(p);
        return cuda_fail(e, "cudaFuncSetAttribute");
    }
    if ((e = cudaMalloc(&p->words, kWords * sizeof(unsigned))) != cudaSuccess ||
        (e = cudaMemset(p->words, 0, kWords * sizeof(unsigned))) != cudaSuccess) {
        free_plan(p);
        return cuda_fail(e, "cudaMalloc(device words)");
    }
    const int sms = prop.multiProcessorCount;
    memset(&p->pre, 0, sizeof p->pre);
    memset(&p->dec, 0, sizeof p->dec);
    if (mode == ROUTE_DECODE) {
        DecodeArgs &a = p->dec;
        a.rows = rows;
        a.timeout_ns = kDefaultTimeoutNs;
        // the plan's column tiles: all 18, or a column shard's
        const int lt = (p->n_lat + kDTileCols - 1) / kDTileCols;
        const int nt = lt + (p->n_exp + kDTileCols - 1) / kDTileCols;
        decode_partition(a, decode_grid(sms, kMaxGrid, nt), &p->segments, lt, nt);
        p->ws_bytes = (size_t)p->segments * kDecodeMaxRows * kDTileCols * sizeof(float2);
        if ((e = cudaMalloc(&p->ws, p->ws_bytes)) != cudaSuccess) {
            free_plan(p);
            return cuda_fail(e, "cudaMalloc(split-K scratch)");
        }
        a.ws = p->ws;
        a.words = p->words;
        p->grid = a.grid;
    } else {
        ProjArgs &a = p->pre;
        a.rows = rows;
        a.timeout_ns = kDefaultTimeoutNs;
        a.n_latent = p->n_lat;
        a.n_experts = p->n_exp;
        a.status = p->words + kWordStatus;
        std::vector<int> off[2], tiles[2];
        for (int ks = 0; ks < 2; ++ks)
            if (!build_schedule(rows, ks == 1, sms / 2, (p->n_lat + 255) / 256,
                                (p->n_exp + 255) / 256, off[ks], tiles[ks], &p->sched_pairs[ks])) {
                free_plan(p);
                return fail(ROUTE_ERR_PLAN, "prefill tile list longer than %d tiles a pair", kMaxPairTiles);
            }
        size_t n = 0;
        for (int ks = 0; ks < 2; ++ks) n += off[ks].size() + tiles[ks].size();
        if ((e = cudaMalloc(&p->sched, n * sizeof(int))) != cudaSuccess) {
            free_plan(p);
            return cuda_fail(e, "cudaMalloc(prefill schedule)");
        }
        size_t at = 0;
        for (int ks = 0; ks < 2 && e == cudaSuccess; ++ks) {
            p->sched_off[ks] = p->sched + at;
            e = cudaMemcpy(p->sched + at, off[ks].data(), off[ks].size() * sizeof(int),
                           cudaMemcpyHostToDevice);
            at += off[ks].size();
            p->sched_tiles[ks] = p->sched + at;
            if (e == cudaSuccess)
                e = cudaMemcpy(p->sched + at, tiles[ks].data(), tiles[ks].size() * sizeof(int),
                               cudaMemcpyHostToDevice);
            at += tiles[ks].size();
        }
        if (e != cudaSuccess) {
            free_plan(p);
            return cuda_fail(e, "copy the prefill schedule");
        }
        // per-row latent sum-of-squares parts (route_step_sumsq; not for shards)
        p->ws_bytes = num_shards ? 0 : (size_t)rows * kSsParts * sizeof(float2);
        if (p->ws_bytes && (e = cudaMalloc(&p->ws, p->ws_bytes)) != cudaSuccess) {
            free_plan(p);
            return cuda_fail(e, "cudaMalloc(sum-of-squares parts)");
        }
        p->segments = (int)tiles[0].size();
        p->grid = 2 * p->sched_pairs[0];
    }
    p->staging_bytes = num_shards ? 0 : staging_size(rows);
    if (p->staging_bytes && (e = cudaMalloc(&p->staging, p->staging_bytes)) != cudaSuccess) {
        free_plan(p);
        return cuda_fail(e, "cudaMalloc(staging)");
    }
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) {
        free_plan(p);
        return cuda_fail(e, "cudaDeviceSynchronize");
    }
    *out = p;
    return ROUTE_OK;
}

}  // namespace

extern "C" {

const char *route_last_error(void) { return g_err; }

route_status route_prepare(int mode, int rows, int device, route_plan **out) {
    return prepare_plan(mode, rows, device, 0, 0, out);
}

route_status route_prepare_shard(int rows, int device, int shard, int num_shards,
                                 route_plan **out) {
    g_err[0] = '\0';
    if (!out) return fail(ROUTE_ERR_NULL, "out is NULL");
    *out = nullptr;
    if (num_shards < 1 || num_shards > kMaxShards || kExperts % num_shards != 0 ||
        kExperts / num_shards < kTopK)
        return fail(ROUTE_ERR_PLAN,
                    "num_shards must divide %d experts and %d latent columns with at least %d "
                    "experts a shard, at most %d shards (1, 2, 4, 7, 8, 14 or 16); got %d",
                    kExperts, kLatent, kTopK, kMaxShards, num_shards);
    if (shard < 0 || shard >= num_shards)
        return fail(ROUTE_ERR_PLAN, "shard %d is not in 0..%d", shard, num_shards - 1);
    // decode sizes stream the shard's weights with split-K over the SMs;
    // larger chunks run the CTA-pair GEMM over the shard's tiles
    return prepare_plan(rows <= ROUTE_DECODE_MAX_ROWS ? ROUTE_DECODE : ROUTE_PREFILL, rows, device,
                        shard, num_shards, out);
}

route_status route_destroy(route_plan *plan) {
    if (!plan) return ROUTE_OK;
    DeviceGuard guard(plan->device);
    cudaDeviceSynchronize();
    free_plan(plan);
    return ROUTE_OK;
}

route_status latent_router_forward(const route_plan *plan, const void *hidden,
                                   const void *W_latent, const void *W_router, void *latent,
                                   float *logits, void *stream) {
    route_status st = check_forward_args(plan, hidden, W_latent, W_router, latent, logits);
    if (st != ROUTE_OK) return st;
    DeviceGuard guard(plan->device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    return launch_forward(plan, hidden, W_latent, W_router, latent, logits, nullptr, nullptr, 0,
                          nullptr,
                          static_cast<cudaStream_t>(stream));
}

route_status topk16_select(const route_plan *plan, const float *logits, int32_t *ids,
                           float *weights, void *stream) {
    route_status st = check_topk_args(plan, logits, ids, weights);
    if (st != ROUTE_OK) return st;
    DeviceGuard guard(plan->device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    cudaError_t e = topk_launch(logits, plan->rows, ids, weights, nullptr, nullptr,
                                static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "top-16 kernel launch");
    return ROUTE_OK;
}

route_status route_step(const route_plan *plan, const void *hidden, const void *W_latent,
                        const void *W_router, void *latent, float *logits, int32_t *ids,
                        float *weights, void *stream) {
    route_status st = check_forward_args(plan, hidden, W_latent, W_router, latent, logits);
    if (st != ROUTE_OK) return st;
    if ((st = check_topk_args(plan, logits, ids, weights)) != ROUTE_OK) return st;
    DeviceGuard guard(plan->device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    return run_step(plan, hidden, W_latent, W_router, latent, logits, ids, weights,
                    static_cast<cudaStream_t>(stream));
}

route_status route_step_sumsq(const route_plan *plan, const void *hidden, const void *W_latent,
                              const void *W_router, void *latent, float *logits, int32_t *ids,
                              float *weights, float *latent_sumsq, void *stream) {
    route_status st = check_forward_args(plan, hidden, W_latent, W_router, latent, logits);
    if (st != ROUTE_OK) return st;
    if ((st = check_topk_args(plan, logits, ids, weights)) != ROUTE_OK) return st;
    if (!latent_sumsq) return fail(ROUTE_ERR_NULL, "latent_sumsq must be non-NULL");
    if ((reinterpret_cast<uintptr_t>(latent_sumsq) & 3u) != 0)
        return fail(ROUTE_ERR_ALIGN, "latent_sumsq must be 4-byte aligned");
    DeviceGuard guard(plan->device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    return run_step(plan, hidden, W_latent, W_router, latent, logits, ids, weights,
                    static_cast<cudaStream_t>(stream), latent_sumsq);
}

route_status route_shard_step(const route_plan *plan, const void *hidden,
                              const void *W_latent_shard, const void *W_router_shard,
                              void *latent_shard, float *logits_shard, int32_t *cand_ids,
                              float *cand_logits, void *stream) {
    route_status st = check_plan(plan);
    if (st != ROUTE_OK) return st;
    if (plan->num_shards == 0)
        return fail(ROUTE_ERR_PLAN, "route_shard_step needs a plan from route_prepare_shard");
    if (!hidden || !W_latent_shard || !W_router_shard || !latent_shard || !logits_shard ||
        !cand_ids || !cand_logits)
        return fail(ROUTE_ERR_NULL, "every pointer must be non-NULL");
    if (!aligned16(hidden) || !aligned16(W_latent_shard) || !aligned16(W_router_shard) ||
        !aligned16(latent_shard) || !aligned16(logits_shard) || !aligned16(cand_ids) ||
        !aligned16(cand_logits))
        return fail(ROUTE_ERR_ALIGN, "every device pointer must be 16-byte aligned");
    DeviceGuard guard(plan->device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (plan->mode == ROUTE_DECODE) {
        CUtensorMap mh, ml, mr;
        if ((st = encode_all(plan, hidden, W_latent_shard, W_router_shard, &mh, &ml, &mr)) !=
            ROUTE_OK)
            return st;
        DecodeArgs a = plan->dec;
        a.latent = static_cast<uint16_t *>(latent_shard);
        a.logits = logits_shard;
        const cudaError_t e = decode_shard_launch(plan->bn, mh, ml, mr, a, plan->n_lat, plan->n_exp,
                                                  plan->shard * plan->n_exp, cand_ids, cand_logits, s);
        return e == cudaSuccess ? ROUTE_OK : cuda_fail(e, "decode shard kernel launch");
    }
    if ((st = launch_forward(plan, hidden, W_latent_shard, W_router_shard, latent_shard,
                             logits_shard, nullptr, nullptr, 0, nullptr, s)) != ROUTE_OK)
        return st;
    const cudaError_t e = shard_topk_launch(logits_shard, plan->rows, plan->n_exp,
                                            plan->shard * plan->n_exp, cand_ids, cand_logits, s);
    return e == cudaSuccess ? ROUTE_OK : cuda_fail(e, "shard top-16 kernel launch");
}

route_status route_merge_candidates(int rows, int num_shards, const int32_t *cand_ids,
                                    const float *cand_logits, int32_t *ids, float *weights,
                                    void *stream) {
    g_err[0] = '\0';
    if (rows < 1 || rows > ROUTE_PREFILL_MAX_ROWS)
        return fail(ROUTE_ERR_ROWS, "rows must be 1-%d; got %d", ROUTE_PREFILL_MAX_ROWS, rows);
    if (num_shards < 1 || num_shards > kMaxShards)
        return fail(ROUTE_ERR_PLAN, "num_shards must be 1-%d; got %d", kMaxShards, num_shards);
    if (!cand_ids || !cand_logits || !ids || !weights)
        return fail(ROUTE_ERR_NULL, "every pointer must be non-NULL");
    if (!aligned16(cand_ids) || !aligned16(cand_logits) || !aligned16(ids) || !aligned16(weights))
        return fail(ROUTE_ERR_ALIGN, "every device pointer must be 16-byte aligned");
    const cudaError_t e = merge_launch(cand_ids, cand_logits, rows, num_shards, ids, weights,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ROUTE_OK : cuda_fail(e, "candidate merge kernel launch");
}

// Device-mapped address of page-locked host memory, or nullptr for memory the
// GPU cannot reach directly (pageable memory takes the copy path).
void *mapped_host(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // clear the (non-sticky) error this query left
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return nullptr;
    return a.devicePointer;
}

// The host path without copies: the staging kernel reads the hidden rows
// through their mapped address (h), the finish kernel writes the results to
// the mapped host buffers.  Enqueued on s; nothing waits.
static route_status enqueue_mapped_step(const route_plan *plan, const void *h,
                                        const void *W_latent, const void *W_router, void *lat,
                                        void *lg, void *ids, void *w, cudaStream_t s) {
    const Staging d = staging_of(plan);
    cudaError_t e;
    if ((e = stage_in_launch(h, d.hidden, (size_t)plan->rows * kHidden * 2, s)) != cudaSuccess)
        return cuda_fail(e, "stage hidden rows");
    // after the staging kernel: no overlap
    return launch_forward(plan, d.hidden, W_latent, W_router, lat, static_cast<float *>(lg),
                          static_cast<int32_t *>(ids), static_cast<float *>(w), 1, nullptr, s,
                          true);
}

route_status route_step_host(const route_plan *plan, const void *hidden_host,
                             const void *W_latent, const void *W_router, void *latent_host,
                             float *logits_host, int32_t *ids_host, float *weights_host,
                             void *stream) {
    route_status st = check_whole_plan(plan);
    if (st != ROUTE_OK) return st;
    if (!hidden_host || !W_latent || !W_router || !latent_host || !logits_host || !ids_host ||
        !weights_host)
        return fail(ROUTE_ERR_NULL, "every pointer must be non-NULL");
    if (!aligned16(W_latent) || !aligned16(W_router))
        return fail(ROUTE_ERR_ALIGN, "weight pointers must be 16-byte aligned");
    DeviceGuard guard(plan->device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Staging d = staging_of(plan);
    const size_t r = (size_t)plan->rows;
    cudaError_t e;
    if (plan->mode == ROUTE_DECODE) {
        // Page-locked host buffers: a staging kernel reads the hidden rows
        // through the mapped address and the finish kernel writes the results
        // straight into the caller's buffers -- no copies to wait for.
        void *h = mapped_host(hidden_host), *lat = mapped_host(latent_host),
             *lg = mapped_host(logits_host), *ids = mapped_host(ids_host),
             *w = mapped_host(weights_host);
        if (h && lat && lg && ids && w && aligned16(h) && aligned16(lat) && aligned16(lg) &&
            aligned16(ids) && aligned16(w)) {
            if ((st = enqueue_mapped_step(plan, h, W_latent, W_router, lat, lg, ids, w, s)) !=
                ROUTE_OK)
                return st;
            if ((e = cudaStreamSynchronize(s)) != cudaSuccess)
                return cuda_fail(e, "cudaStreamSynchronize");
            return ROUTE_OK;
        }
    }
    if ((e = cudaMemcpyAsync(d.hidden, hidden_host, r * kHidden * 2, cudaMemcpyHostToDevice, s)) !=
        cudaSuccess)
        return cuda_fail(e, "copy hidden to device");
    if ((st = launch_forward(plan, d.hidden, W_latent, W_router, d.latent, d.logits, d.ids,
                             d.weights, 1, nullptr, s, true)) != ROUTE_OK)
        return st;
    if ((e = cudaMemcpyAsync(latent_host, d.latent, r * kLatent * 2, cudaMemcpyDeviceToHost, s)) !=
            cudaSuccess ||
        (e = cudaMemcpyAsync(logits_host, d.logits, r * kExperts * 4, cudaMemcpyDeviceToHost, s)) !=
            cudaSuccess ||
        (e = cudaMemcpyAsync(ids_host, d.ids, r * kTopK * 4, cudaMemcpyDeviceToHost, s)) !=
            cudaSuccess ||
        (e = cudaMemcpyAsync(weights_host, d.weights, r * kTopK * 4, cudaMemcpyDeviceToHost, s)) !=
            cudaSuccess)
        return cuda_fail(e, "copy results to host");
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return ROUTE_OK;
}

route_status route_device_status(const route_plan *plan) {
    route_status st = check_plan(plan);
    if (st != ROUTE_OK) return st;
    DeviceGuard guard(plan->device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    unsigned status = 0;
    if ((e = cudaMemcpy(&status, plan->words, sizeof status, cudaMemcpyDeviceToHost)) !=
        cudaSuccess)
        return cuda_fail(e, "read device status");
    if (status == 0) return ROUTE_OK;
    cudaMemset(plan->words, 0, kWords * sizeof(unsigned));  // the status word area
    cudaDeviceSynchronize();
    if (status & kStatusBounds)
        return fail(ROUTE_ERR_DEVICE_BOUNDS,
                    "a kernel computed an index out of range and skipped that access (status "
                    "0x%x, debug library); that launch's outputs are invalid",
                    status);
    return fail(ROUTE_ERR_DEVICE_TIMEOUT,
                "a kernel gave up waiting (status 0x%x); that launch's outputs are invalid", status);
}

route_status route_host_step_create(route_plan *plan, const void *hidden_host,
                                    const void *W_latent, const void *W_router,
                                    void *latent_host, float *logits_host, int32_t *ids_host,
                                    float *weights_host, void *stream, route_host_step **out) {
    route_status st = check_plan(plan);
    if (st != ROUTE_OK) return st;
    if (!out) return fail(ROUTE_ERR_NULL, "out must be non-NULL");
    *out = nullptr;
    if (!hidden_host || !W_latent || !W_router || !latent_host || !logits_host || !ids_host ||
        !weights_host)
        return fail(ROUTE_ERR_NULL, "every pointer must be non-NULL");
    if (!aligned16(W_latent) || !aligned16(W_router))
        return fail(ROUTE_ERR_ALIGN, "weight pointers must be 16-byte aligned");
    if (plan->mode != ROUTE_DECODE || plan->num_shards != 0)
        return fail(ROUTE_ERR_PLAN, "host steps are prepared for decode plans only");
    DeviceGuard guard(plan->device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    void *h = mapped_host(hidden_host), *lat = mapped_host(latent_host),
         *lg = mapped_host(logits_host), *ids = mapped_host(ids_host),
         *w = mapped_host(weights_host);
    if (!(h && lat && lg && ids && w && aligned16(h) && aligned16(lat) && aligned16(lg) &&
          aligned16(ids) && aligned16(w)))
        return fail(ROUTE_ERR_PLAN,
                    "host steps need every host buffer page-locked and 16-byte aligned");
    route_host_step *step = new (std::nothrow) route_host_step{};
    if (!step) return fail(ROUTE_ERR_CUDA, "out of host memory");
    step->stream = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMalloc(&step->counter, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemset(step->counter, 0, sizeof(unsigned));
    if (e == cudaSuccess)
        e = cudaHostAlloc(reinterpret_cast<void **>(&step->flag_host), 64, cudaHostAllocMapped);
    if (e == cudaSuccess) {
        *step->flag_host = 0u;
        e = cudaHostGetDevicePointer(reinterpret_cast<void **>(&step->flag_dev), step->flag_host, 0);
    }
    // the direct launches' two staging buffers, then the `published` word
    step->hbuf_stride = align256((size_t)plan->rows * kHidden * 2);
    if (e == cudaSuccess) e = cudaMalloc(&step->hbuf, 2 * step->hbuf_stride + 256);
    if (e == cudaSuccess) {
        step->published = reinterpret_cast<unsigned *>(step->hbuf + 2 * step->hbuf_stride);
        e = cudaMemset(step->published, 0, sizeof(unsigned));
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();  // the counter's zero is in place
    // Capture on a stream of our own: the caller's may be the legacy
    // default stream, which cannot be captured.
    cudaStream_t cs = nullptr;
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
        st = enqueue_mapped_step(plan, h, W_latent, W_router, lat, lg, ids, w, cs);
        if (st == ROUTE_OK) {
            const cudaError_t e3 = host_done_launch(step->counter, step->flag_dev, cs);
            if (e3 != cudaSuccess) st = cuda_fail(e3, "completion kernel launch");
        }
        const cudaError_t e2 = cudaStreamEndCapture(cs, &step->graph);
        if (st == ROUTE_OK && e2 != cudaSuccess) e = e2;
    }
    if (st == ROUTE_OK && e == cudaSuccess)
        e = cudaGraphInstantiate(&step->exec, step->graph, 0);
    if (cs) cudaStreamDestroy(cs);
    if (st != ROUTE_OK || e != cudaSuccess) {
        release_step_graph(step);
        delete step;
        return st != ROUTE_OK ? st : cuda_fail(e, "capture the host step");
    }
    for (int j = 0; j < 2 && st == ROUTE_OK; ++j)
        st = encode_2d(&step->hmap[j], step->hbuf + j * step->hbuf_stride, kHidden,
                       (uint64_t)plan->rows, kKBlock, (uint32_t)plan->bn, "hidden");
    if (st != ROUTE_OK) {
        release_step_graph(step);
        delete step;
        return st;
    }
    step->hidden_mapped = h;
    step->W_latent = W_latent;
    step->W_router = W_router;
    step->dec = plan->dec;
    step->dec.latent = static_cast<uint16_t *>(lat);
    step->dec.logits = static_cast<float *>(lg);
    step->dec.ids = static_cast<int32_t *>(ids);
    step->dec.weights = static_cast<float *>(w);
    step->dec.sumsq = nullptr;
    step->dec.overlap = 0;  // after the staging kernel
    step->plan = plan;
    step->next = plan->steps;
    plan->steps = step;
    *out = step;
    return ROUTE_OK;
}

// The step's kernels launched one by one on its stream, each chained to its
// predecessor by programmatic dependent launch: a staging kernel that copies
// the hidden rows into the step's next buffer (once the launch that last read
// that buffer has finished) and publishes them, the stream kernel in overlap
// mode, which reads them as soon as they are published -- under the tail of
// whatever precedes it on the stream, typically another step -- and writes
// scratch only after that has finished, the finish kernel and the completion
// kernel.
static route_status enqueue_host_step(route_host_step *step) {
    const route_plan *p = step->plan;
    const unsigned launch = step->launched + 1u;
    const int j = (int)(step->staged & 1u);
    int ctas = 0;
    cudaError_t e = stage_publish_launch(
        step->hidden_mapped, step->hbuf + j * step->hbuf_stride, (size_t)p->rows * kHidden * 2,
        step->counter, step->buf_launch[j], step->published, p->words, step->dec.timeout_ns, &ctas,
        step->stream);
    if (e != cudaSuccess) return cuda_fail(e, "stage hidden rows");
    // the rows are on their way into buffer j: count them even if a launch
    // below fails (the device adds them all the same)
    step->published_total += (unsigned)ctas;
    step->staged += 1u;
    step->buf_launch[j] = launch;
    CUtensorMap ml, mr;
    route_status st;
    if ((st = cached_map(p->map_wl, step->W_latent, (uint64_t)p->n_lat, kHidden, 64, kKBlock,
                         "W_latent", &ml)) != ROUTE_OK ||
        (st = cached_map(p->map_wr, step->W_router, (uint64_t)p->n_exp, kHidden, 64, kKBlock,
                         "W_router", &mr)) != ROUTE_OK)
        return st;
    DecodeArgs a = step->dec;
    a.overlap = 1;
    a.hidden_count = step->published;
    a.hidden_target = step->published_total;
    if ((e = decode_launch(p->bn, step->hmap[j], ml, mr, a, 1, step->stream)) != cudaSuccess)
        return cuda_fail(e, "decode kernel launch");
    if ((e = host_done_launch(step->counter, step->flag_dev, step->stream)) != cudaSuccess)
        return cuda_fail(e, "completion kernel launch");
    return ROUTE_OK;
}

// True when another step of the plan has a launch in flight on a stream
// other than this step's: the two would share the plan's scratch unordered.
static bool in_flight_elsewhere(const route_host_step *step) {
    for (const route_host_step *o = step->plan->steps; o; o = o->next) {
        if (o == step || o->stream == step->stream || !o->flag_host) continue;
        const unsigned v = __atomic_load_n(o->flag_host, __ATOMIC_ACQUIRE);
        if ((int)(v - o->launched) < 0) return true;
    }
    return false;
}

route_status route_host_step_launch(route_host_step *step) {
    g_err[0] = '\0';
    if (!step || !step->plan || !step->exec)
        return fail(ROUTE_ERR_NULL, "host step is NULL or its plan has been destroyed");
    if (in_flight_elsewhere(step))
        return fail(ROUTE_ERR_PLAN, "another step of this plan is in flight on another stream");
    DeviceGuard guard(step->plan->device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    const route_status st = enqueue_host_step(step);
    if (st != ROUTE_OK) return st;
    ++step->launched;
    return ROUTE_OK;
}

route_status route_host_step_wait(route_host_step *step) {
    g_err[0] = '\0';
    if (!step || !step->plan || !step->exec)
        return fail(ROUTE_ERR_NULL, "host step is NULL or its plan has been destroyed");
    // Wait for the latest launch's number in the completion word (the
    // results are in host memory before it); after kHostWaitNs without it,
    // wait for the stream instead and report what it reports.  Every return
    // leaves no launch of this step unfinished (the wait ends on the latest
    // number, or after the stream has drained), and `done` takes the word's
    // value then.
    const unsigned want = step->launched;
    auto reached = [&](unsigned v) { return (int)(v - want) >= 0; };
    if (reached(step->done)) return ROUTE_OK;  // nothing in flight
    const auto t0 = std::chrono::steady_clock::now();
    for (uint32_t it = 1;; ++it) {
        const unsigned v = __atomic_load_n(step->flag_host, __ATOMIC_ACQUIRE);
        if (reached(v)) {
            step->done = v;
            return ROUTE_OK;
        }
        if ((it & 1023u) == 0u &&
            std::chrono::steady_clock::now() - t0 > std::chrono::nanoseconds(kHostWaitNs))
            break;
    }
    DeviceGuard guard(step->plan->device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    cudaError_t e = cudaStreamSynchronize(step->stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    const unsigned v = __atomic_load_n(step->flag_host, __ATOMIC_ACQUIRE);
    step->done = step->launched = v;  // nothing of this step is in flight now
    if (!reached(v))
        return fail(ROUTE_ERR_DEVICE, "the host step finished without its completion word");
    return ROUTE_OK;
}

route_status route_host_step_run(route_host_step *step) {
    g_err[0] = '\0';
    if (!step || !step->plan || !step->exec)
        return fail(ROUTE_ERR_NULL, "host step is NULL or its plan has been destroyed");
    if (in_flight_elsewhere(step))
        return fail(ROUTE_ERR_PLAN, "another step of this plan is in flight on another stream");
    {
        DeviceGuard guard(step->plan->device);
        if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
        const cudaError_t e = cudaGraphLaunch(step->exec, step->stream);
        if (e != cudaSuccess) return cuda_fail(e, "launch the host step");
        ++step->launched;
    }
    return route_host_step_wait(step);
}

route_status route_host_step_destroy(route_host_step *step) {
    if (!step) return ROUTE_OK;
    if (route_plan *p = step->plan) {
        for (route_host_step **q = &p->steps; *q; q = &(*q)->next)
            if (*q == step) {
                *q = step->next;
                break;
            }
        DeviceGuard guard(p->device);
        cudaStreamSynchronize(step->stream);  // its last launch may still be leaving
        release_step_graph(step);
    }
    delete step;
    return ROUTE_OK;
}

route_status route_set_overlap(route_plan *plan, int enable) {
    route_status st = check_plan(plan);
    if (st != ROUTE_OK) return st;
    plan->dec.overlap = plan->pre.overlap = enable ? 1 : 0;
    return ROUTE_OK;
}

route_status route_set_latent_ksplit(route_plan *plan, int enable) {
    route_status st = check_plan(plan);
    if (st != ROUTE_OK) return st;
    if (plan->mode == ROUTE_PREFILL) {  // K slices of 14 k-blocks split every prefill tile evenly
        plan->pre_ksplit = enable ? 1 : 0;
        return ROUTE_OK;
    }
    if (plan->num_shards != 0 && enable)
        return fail(ROUTE_ERR_PLAN, "a decode-size column shard has no K-split latent");
    if (enable) {
        // every CTA that touches a latent tile must own exactly one K slice of it
        constexpr int kSlice = kKBlocks / kKSplitSlices;  // 14 k-blocks = 896 of K
        const DecodeArgs &a = plan->dec;
        for (int g = 0; g < a.grid; ++g) {
            const int u0 = a.cta_unit[g], u1 = a.cta_unit[g + 1];
            if (u0 >= kDLatTiles * kKBlocks) break;
            if (u0 % kSlice != 0 || u1 - u0 != kSlice)
                return fail(ROUTE_ERR_PLAN,
                            "this device's split-K partition (%d CTAs) does not align with the %d "
                            "K slices the K-split latent needs",
                            a.grid, kKSplitSlices);
        }
    }
    plan->dec.ksplit = enable ? 1 : 0;
    return ROUTE_OK;
}

route_status route_test_stall(route_plan *plan, int enable, uint64_t timeout_ns) {
    route_status st = check_plan(plan);
    if (st != ROUTE_OK) return st;
    const unsigned long long t = enable ? (timeout_ns ? timeout_ns : 1000000ull) : kDefaultTimeoutNs;
    plan->pre.test_stall = plan->dec.test_stall = enable ? 1 : 0;
    plan->pre.timeout_ns = plan->dec.timeout_ns = t;
    return ROUTE_OK;
}

route_status route_test_poison_scratch(const route_plan *plan, void *stream) {
    route_status st = check_plan(plan);
    if (st != ROUTE_OK) return st;
    if (!plan->ws) return ROUTE_OK;
    DeviceGuard guard(plan->device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    const cudaError_t e =
        cudaMemsetAsync(plan->ws, 0xFF, plan->ws_bytes, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ROUTE_OK : cuda_fail(e, "poison the scratch");
}

route_status route_step_decode_noalloc(int rows, const void *hidden, const void *W_latent,
                                       const void *W_router, void *latent, float *logits,
                                       int32_t *ids, float *weights, void *stream) {
    g_err[0] = '\0';
    if (rows < 1 || rows > ROUTE_DECODE_MAX_ROWS)
        return fail(ROUTE_ERR_ROWS,
                    "route_step_decode_noalloc handles 1-%d rows (its fixed scratch is sized for "
                    "%d); got %d",
                    ROUTE_DECODE_MAX_ROWS, ROUTE_DECODE_MAX_ROWS, rows);
    if (!hidden || !W_latent || !W_router || !latent || !logits || !ids || !weights)
        return fail(ROUTE_ERR_NULL, "every pointer must be non-NULL");
    if (!aligned16(hidden) || !aligned16(W_latent) || !aligned16(W_router) || !aligned16(latent) ||
        !aligned16(logits) || !aligned16(ids) || !aligned16(weights))
        return fail(ROUTE_ERR_ALIGN, "every device pointer must be 16-byte aligned");
    int device = -1;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (device < 0 || device >= kNoAllocMaxDevices)
        return fail(ROUTE_ERR_DEVICE, "device %d is out of range", device);
    NoAllocDevice *d = nullptr;
    route_status st = noalloc_setup(device, &d);
    if (st != ROUTE_OK) return st;
    const int bn = decode_bn_for(rows);
    CUtensorMap mh, ml, mr;
    if ((st = encode_2d(&mh, hidden, kHidden, (uint64_t)rows, kKBlock, (uint32_t)bn, "hidden")) !=
            ROUTE_OK ||
        (st = encode_2d(&ml, W_latent, kLatent, kHidden, 64, kKBlock, "W_latent")) != ROUTE_OK ||
        (st = encode_2d(&mr, W_router, kExperts, kHidden, 64, kKBlock, "W_router")) != ROUTE_OK)
        return st;
    DecodeArgs a = d->base;
    a.rows = rows;
    a.latent = static_cast<uint16_t *>(latent);
    a.logits = logits;
    a.ids = ids;
    a.weights = weights;
    e = decode_launch(bn, mh, ml, mr, a, 1, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
    return ROUTE_OK;
}

route_status route_noalloc_status(int device) {
    g_err[0] = '\0';
    if (device < 0 || device >= kNoAllocMaxDevices)
        return fail(ROUTE_ERR_DEVICE, "device %d is out of range", device);
    unsigned char *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (g_noalloc[device].ready) scratch = g_noalloc[device].scratch;
    }
    if (!scratch) return ROUTE_OK;  // no call has run on this device
    DeviceGuard guard(device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    unsigned status = 0;
    if ((e = cudaMemcpy(&status, scratch, sizeof status, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "read the no-allocation status word");
    if (status == 0) return ROUTE_OK;
    if ((e = cudaMemset(scratch, 0, kNoAllocWordBytes)) != cudaSuccess ||
        (e = cudaDeviceSynchronize()) != cudaSuccess)
        return cuda_fail(e, "clear the no-allocation status");
    return fail(ROUTE_ERR_DEVICE_TIMEOUT,
                "a kernel of route_step_decode_noalloc gave up waiting (status 0x%x); that call's "
                "outputs are invalid",
                status);
}

route_status route_test_noalloc_stall(int device, int enable, uint64_t timeout_ns) {
    g_err[0] = '\0';
    if (device < 0 || device >= kNoAllocMaxDevices)
        return fail(ROUTE_ERR_DEVICE, "device %d is out of range", device);
    DeviceGuard guard(device);
    if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
    NoAllocDevice *d = nullptr;
    route_status st = noalloc_setup(device, &d);
    if (st != ROUTE_OK) return st;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    d->base.test_stall = enable ? 1 : 0;
    d->base.timeout_ns = enable ? (timeout_ns ? timeout_ns : 1000000ull) : kDefaultTimeoutNs;
    return ROUTE_OK;
}

int route_noalloc_grid(int device) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return decode_grid(prop.multiProcessorCount, kNoAllocMaxGrid);
}

int route_plan_rows(const route_plan *plan) { return plan ? plan->rows : -1; }
int route_plan_mode(const route_plan *plan) { return plan ? plan->mode : -1; }
int route_plan_grid(const route_plan *plan) { return plan ? plan->grid : -1; }
int route_plan_segments(const route_plan *plan) { return plan ? plan->segments : -1; }
int route_plan_latent_cols(const route_plan *plan) { return plan ? plan->n_lat : -1; }
int route_plan_experts(const route_plan *plan) { return plan ? plan->n_exp : -1; }

}  // extern "C"
