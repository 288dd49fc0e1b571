// Grouped tcgen05 GEMM of the expert FFN (and of the router's tensor-core
// logits): tile shapes, the tile list, the launch arguments.  Internal, not
// part of the C ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace moe {

// Status word bits (mirrors include/moe_api.h).
constexpr int kDevErrExpertRange = 0x1;
constexpr int kDevErrTimeout = 0x2;
constexpr int kDevErrBadBlocks = 0x4;
// Calls whose tiles hold at most this many routed rows run the CTA-pair
// GEMMs' decode instances (the small-tile token box of the other instances).
constexpr int kDecodeMaxT = 32;
constexpr int kDevNoteRerouteFallback = 0x100;

// Rows of one grouped-GEMM token tile (the N of every tcgen05 MMA), one
// fixed value per GEMM for every layer and every T: one tile shape, one K
// order.  W2 takes 256-row tiles (fewer shared-memory bytes per flop); W13
// keeps 128 rows so that its gate and up accumulators stay double-buffered in
// the 512 TMEM columns and the epilogue overlaps the next tile's MMAs; the
// router's tensor-core logits use 128.
constexpr int kW13TileRows = 128;
constexpr int kW2TileRows = 256;
constexpr int kRouterTileRows = 128;
// The router's logits in 64-row token tiles when 128-row tiles would leave
// SMs idle: they only filter candidates (every output logit is recomputed in
// the canonical order), so the tile height may follow the batch.
constexpr int kRouterTileRowsNarrow = 64;
constexpr int kMaxTileRows = 256;
// Output features of one grouped-GEMM tile (the M of every MMA).
constexpr int kTileFeat = 128;

struct GemmTile {
  int32_t expert;
  int32_t row0;   // first padded row of the tile
  int32_t rows;   // padded rows of the expert's segment in this tile (<= the tile size)
  int32_t first;  // index of the first tile of this expert in the list
  int32_t count;  // tiles of this expert
  int32_t valid;  // rows holding a route: rows [row0, row0 + valid) (<= rows); the rest is padding
  int32_t pad[2];
};

// ---- grouped expert GEMMs (tcgen05)
struct GemmArgs {
  int K;               // reduction length (H for W13, I for W2)
  int n_feat_tiles;    // output features / kTileFeat (I for W13, H for W2)
  int w_rows_per_e;    // rows of one expert in the 2-D weight map (= K)
  int up_col;          // column offset of the "up" half in W13 (= I)
  const GemmTile* tiles;     // routed mode: tile list on the device
  const int32_t* num_tiles;  // routed mode: device count
  int identity_T;            // identity mode (shared expert): rows 0..T-1, else 0
  void* out;           // W13: bf16 a [rows, I]; W2: y [rows, H] (bf16 with out_bf16, else fp32);
                       // router logits: fp32 [T, N]
  int out_ld;          // elements per output row
  int* status;
  int out_bf16;        // non-W13 outputs rounded to bf16 (the expert outputs y), else fp32
  int concurrent;      // work units resident at once (set by the launcher)
  int pair;            // 1: CTA-pair kernel (256 token rows per tile, token maps with
                       //    128-row boxes; n_feat_tiles in units of kPairFeatW13 / kPairFeatW2)
  int wide;            // W2 pairs only, 1: items of two 256-feature groups
                       //    (n_feat_tiles in units of kPairFeatW2Wide)
  int decode;          // pairs only, 1: every tile holds at most 32 routed rows (the
                       //    caller's batch has at most 32 tokens); stages then hold a
                       //    32-row token box, so more of them fit

  unsigned long long wait_ns;  // limit of the pipeline waits; 0: kWaitLimitNs
  int32_t* next_item;  // one-CTA kernel, routed mode: the launch's tile counter (zero before the
                       // launch); each CTA takes the next item from it when it is free.  nullptr
                       // (and the pair kernels): CTA (pair) u takes items u, u + grid, ...  Only
                       // which CTA runs a tile changes, never the tile's arithmetic.
};

// Rows of a CTA-pair token tile, the token box each CTA of the pair loads,
// and the output features of one pair tile.
constexpr int kPairTileRows = 256;
constexpr int kPairBoxRows = 128;
constexpr int kPairFeatW13 = 128;
constexpr int kPairFeatW2 = 256;
// Whether a GEMM with this many output features and reduction length K runs
// on CTA pairs: a property of the layer's shape, never of T.
bool gemm_pair_ok(bool w13, int features, int K);
// Whether the W2 pairs take wide items (two 256-feature groups on one token
// tile): a long reduction and 512 | features, a property of the layer.
constexpr int kPairFeatW2Wide = 512;
constexpr int kWideMinK = 8192;
bool gemm_wide_ok(int features, int K);

bool gemm_smem_ok();
// x_small: the same token tensor with a 32-row box (tiles with <= 32 rows)
void launch_w13_gemm(const CUtensorMap& w_map, const CUtensorMap& x_map, const CUtensorMap& x_small,
                     const GemmArgs& a, int max_tiles, int num_sms, cudaStream_t s);
void launch_w2_gemm(const CUtensorMap& w_map, const CUtensorMap& x_map, const CUtensorMap& x_small,
                    const GemmArgs& a, int max_tiles, int num_sms, cudaStream_t s);
void launch_router_gemm(const CUtensorMap& w_map, const CUtensorMap& x_map, const CUtensorMap& x_small,
                        const GemmArgs& a, int max_tiles, int num_sms, cudaStream_t s, int tile_rows);

}  // namespace moe
