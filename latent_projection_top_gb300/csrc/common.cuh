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

// Tiling of the projection: one tile = 128 weight columns (the MMA M side)
// x BN token rows (the MMA N side); K is consumed 64 at a time.
constexpr int kTileCols = 128;
constexpr int kKBlock = 64;
constexpr int kKBlocks = kHidden / kKBlock;                 // 112
constexpr int kLatentTiles = kLatent / kTileCols;           // 28
constexpr int kRouterTiles = kExperts / kTileCols;          // 7
constexpr int kColTiles = kLatentTiles + kRouterTiles;      // 35
constexpr int kProjThreads = 192;                           // 6 warps

enum Mode : int { kDecode = 0, kPrefill = 1 };

// Device status bits (the kernels set them instead of hanging).
constexpr unsigned kStatusTimeout = 1u;

// Everything the projection kernel needs besides its three tensor maps.
struct ProjArgs {
    int rows;            // token rows in this call
    int mode;            // kDecode or kPrefill
    int row_tiles;       // prefill: ceil(rows / BN); decode: 1
    int grid;            // CTAs launched
    int units;           // decode: kColTiles * kKBlocks (k-block units split over CTAs)
    int fuse_topk;       // decode: the CTA finishing the last router tile runs the top-16
    int test_stall;      // test hook: skip each CTA's last copy so a wait must time out
    unsigned long long timeout_ns;  // bound on every wait inside the kernel
    // decode split-K partition, fixed at plan time (depends on grid only):
    int seg_base[kColTiles];   // first partial slot of column tile c
    int seg_count[kColTiles];  // number of CTAs (partials) covering tile c
    int cta_first[kColTiles];  // first CTA covering tile c
    float *ws;                 // partials [slot][kDecodeMaxRows][kTileCols] FP32
    unsigned *counters;        // [kColTiles] arrivals per tile, [kColTiles] router tiles done
    unsigned *status;          // device status word
    uint16_t *latent;          // [rows, 3584] BF16 bits
    float *logits;             // [rows, 896]
    int32_t *ids;              // [rows, 16]   (fused top-16 only)
    float *weights;            // [rows, 16]   (fused top-16 only)
};

// Internal launchers (defined next to their kernels).
int proj_bn_for(int mode, int rows);
int proj_smem_bytes(int bn);
cudaError_t proj_configure(int bn);  // opt in to the kernel's shared memory size
cudaError_t proj_launch(int bn, const CUtensorMap &map_h, const CUtensorMap &map_wl,
                        const CUtensorMap &map_wr, const ProjArgs &args, cudaStream_t stream);
cudaError_t topk_launch(const float *logits, int rows, int32_t *ids, float *weights,
                        cudaStream_t stream);

}  // namespace route
