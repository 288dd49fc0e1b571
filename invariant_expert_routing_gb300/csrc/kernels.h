// Internal launchers of the MoE layer kernels (not part of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "gemm.h"

namespace moe {

// Which of several equivalent kernel paths a call takes, and the limit of the
// bounded device waits: moe_config's debug fields (mirrors MOE_DEBUG_* of
// include/moe_api.h).  Zero everywhere: the defaults.  No option changes a
// result bit.
constexpr uint32_t kPathRouterTc = 0x1;
constexpr uint32_t kPathRouterChunked = 0x2;
constexpr uint32_t kPathRowGather = 0x4;
constexpr uint32_t kPathRowScatter = 0x8;
constexpr uint32_t kPathNoDecodeFront = 0x10;
constexpr uint32_t kPathRerouteSequential = 0x20;
constexpr uint32_t kPathRerouteGrid = 0x40;
constexpr uint32_t kPathRerouteOneCta = 0x80;
constexpr uint32_t kPathRouterTile128 = 0x100;
constexpr uint32_t kPathRouterTile64 = 0x200;
struct PathOpts {
  uint32_t flags = 0;
  int grid_ctas = 0;      // > 0: cap on the CTAs of the reroute's grid-wide rounds
  uint64_t wait_ns = 0;   // > 0: limit of the bounded waits (else each wait's default)
};

// Router reduction chunk (elements of H summed in order before combining).
constexpr int kRouterChunk = 256;
// Routes handled by one CTA of the dispatch count/scatter kernels.
constexpr int kDispatchTile = 1024;

// ---- router
// Chunked CUDA-core router: chunk sums in parallel over (chunk, experts,
// tokens), then logits in the canonical chunked order (optional), top-k and
// gates (optional: topk_idx null for logits alone).  Used for at most
// kDecodeRouterMaxT tokens, and for batches unless the tensor-core router
// serves the call and T * H * N exceeds 3 * 2^28.  part:
// chunked_router_part_floats floats.
constexpr int kDecodeRouterMaxT = 64;
bool chunked_router_ok(int T, int H, int N, bool tc_router, uint32_t path_flags);
size_t chunked_router_part_floats(int T, int H, int N);
// the chunk sums alone (part: chunked_router_part_floats floats)
void launch_router_partials(const uint16_t* h, const uint16_t* w_gate, float* part, int T, int H, int N,
                            cudaStream_t s);
void launch_router_chunked(const uint16_t* h, const uint16_t* w_gate, const float* bias, float* part,
                           float* logits, int32_t* topk_idx, float* gates, int T, int H, int N, int k,
                           cudaStream_t s);
// tensor-core router with a certified candidate filter (N % 128 == 0)
void launch_gate_prep(const uint16_t* w_gate, uint16_t* wgT, float* norm_w, int H, int N,
                      cudaStream_t s);
float router_cert_beta(int H);
bool route_certified_ok(int H);
// filter, tiled recompute of the candidates' chunk sums, finalize (three
// launches); scratch: route_certified_scratch_floats floats
size_t route_certified_scratch_floats(int T, int H);
void launch_route_certified(const float* logits_tc, const float* bias, const uint16_t* h,
                            const uint16_t* wgT, const float* norm_w, int T, int H, int N, int k,
                            int32_t* topk_idx, float* gates, int32_t* n_cand, float* scratch,
                            cudaStream_t s);

// ---- dispatch / alignment
// expert_offset (nullable, [N]): for one shard of a larger batch, the routes
// each expert received in the earlier shards; the shard's routes then get
// capacity - expert_offset[e] (at least 0) of expert e's capacity.
void launch_dispatch(const int32_t* topk_idx, int T, int N, int k, int B, int capacity,
                     uint8_t* route_kept, int32_t* route_pos, int32_t* sorted_route_ids,
                     int32_t* block_expert, int32_t* num_padded, int32_t* expert_counts,
                     int32_t* num_dropped, int32_t* rank_in_tile, int32_t* tile_count,
                     int32_t* seg_off, int* status, cudaStream_t s, const int32_t* expert_offset = nullptr);
// Scratch of the overflow reroute (R routes, N experts).
constexpr int kRerouteListLen = 128;  // cached best experts per token with an overflowing slot
// ints of one buffer of the per-round exchange of the grid-wide reroute
// rounds with G CTAs: 16-bit counts [N + 2][G rounded up to 8] (candidates
// per expert, then unplaceable and listed routes), and the exclusive prefix
// of the candidate counts over experts [G][N].
__host__ __device__ inline size_t reroute_exchange_ints(int G, int N) {
  const size_t gs = (size_t)(G + 7) / 8 * 8;
  return ((size_t)(N + 2) * gs / 2 + (size_t)G * N + 3) / 4 * 4;
}
struct RerouteScratch {
  int32_t* list;    // [R] overflowing route ids, ascending
  int32_t* hold;    // [R] per list position: expert held, -1 none, -2 none possible
  int32_t* cand;    // [R] per list position: this round's candidate
  int32_t* ptr;     // [R] per list position: next cached preference to try
  int32_t* first;   // [R] per list position: list position of the token's first overflowing slot
  uint8_t* prefs;   // [T * kRerouteListLen] cached preferences, by token
  int32_t* acc;     // [N] overflowing routes each expert holds at the end
  int32_t* worst;   // [N] largest route id each expert holds (-1 none)
  int32_t* flag;    // [1] non-zero: recompute with the sequential kernel
  int32_t* count;   // [1] overflowing routes
  // grid-wide version (many overflowing routes)
  uint32_t* gsync;  // [4] barrier arrivals, generation, error
  int32_t* lcount;  // [2][reroute_exchange_ints(CTAs, N)] per-CTA counts exchanged each round
  int32_t* lrank;   // [2][R] per-CTA candidate route ids ordered by (expert, rank)
};
// phase two of the reroute: route_expert for every route (kept: its expert,
// overflowing: its new expert or -1), num_dropped / num_rerouted
void launch_reroute(const int32_t* topk_idx, const float* logits, int T, int N, int k, int capacity,
                    const int32_t* rank_in_tile, const int32_t* tile_base, const int32_t* kept_count,
                    const RerouteScratch& sc, int32_t* route_expert, int32_t* num_dropped,
                    int32_t* num_rerouted, int* status, const PathOpts& o, cudaStream_t s);
// phase one of launch_dispatch, overflow reroute, then the layout of the
// final assignment (route_expert: expert per route, -1 = dropped)
void launch_dispatch_reroute(const int32_t* topk_idx, const float* logits, int T, int N, int k, int B,
                             int capacity, uint8_t* route_kept, int32_t* route_expert,
                             int32_t* route_pos, int32_t* sorted_route_ids, int32_t* block_expert,
                             int32_t* num_padded, int32_t* expert_counts, int32_t* num_dropped,
                             int32_t* num_rerouted, int32_t* rank_in_tile, int32_t* tile_count,
                             int32_t* seg_off, const RerouteScratch& sc, int* status, const PathOpts& o,
                             cudaStream_t s);
// stable layout of routes that already carry their expert (-1 = none)
void launch_dispatch_routes(const int32_t* route_expert, int R, int N, int B, uint8_t* route_kept,
                            int32_t* route_pos, int32_t* sorted_route_ids, int32_t* block_expert,
                            int32_t* num_padded, int32_t* expert_counts, int32_t* rank_in_tile,
                            int32_t* tile_count, int32_t* seg_off, int* status, cudaStream_t s);
// expert choice: scores, per-expert top-C selection and the padded layout
void launch_expert_choice(const float* logits, int T, int N, int C, int B, unsigned long long* keys,
                          float* gates, uint8_t* route_kept, int32_t* route_pos, int32_t* sorted_route_ids,
                          int32_t* block_expert, int32_t* num_padded, int32_t* expert_counts,
                          cudaStream_t s);
// a batch of at most 1024 routes: launch_dispatch + both tile lists of launch_tiles_and_rows
// (tile_rows rows_a and rows_b) in one launch, the same integers
bool dispatch_small_ok(long long R);
struct TileListOut;
void launch_dispatch_small(const int32_t* topk_idx, int R, int N, int B, int capacity, uint8_t* route_kept,
                           int32_t* route_pos, int32_t* sorted_route_ids, int32_t* block_expert,
                           int32_t* num_padded, int32_t* expert_counts, int32_t* num_dropped,
                           const TileListOut& la, const TileListOut& lb, int* status, cudaStream_t s);
// decode front (at most 2 tokens, token choice): the router's chunk sums
// (launch_router_partials), then in one CTA the logits in the canonical
// order, top-k and gates, launch_dispatch_small's results and the routed
// token rows of x_perm (padding rows untouched): two launches.
bool decode_front_ok(int T, int H, int N, int k, uint32_t path_flags);
void launch_decode_front(const uint16_t* h, const uint16_t* w_gate, const float* bias, float* part, int T, int H,
                         int N, int k,
                         int B, int capacity, int32_t* topk_idx, float* gates, uint8_t* route_kept,
                         int32_t* route_pos, int32_t* sorted_route_ids, int32_t* block_expert, int32_t* num_padded,
                         int32_t* expert_counts, int32_t* num_dropped, const TileListOut& la,
                         const TileListOut& lb, uint16_t* x_perm, int64_t max_rows, int* status, cudaStream_t s);
// Tile list of one GEMM: tile_rows-row tiles over each expert's padded
// segment; a tile's valid rows end at the segment's last route (sorted ids
// in [0, R)).
struct TileListOut {
  GemmTile* tiles;
  int32_t* num_tiles;
  int tile_rows;
  int max_tiles;
  int32_t* next_item;   // the GEMM's tile counter: zeroed where num_tiles is written
};
// Tiles of one expert segment of `padded` rows (the first `valid` hold
// routes), cut into tile_rows-row tiles from the segment's start.  Tile j of
// nt: rows from row0 + j * tile_rows; the last runs to the segment's end.
__host__ __device__ inline int segment_tiles(int padded, int tile_rows) {
  return (padded + tile_rows - 1) / tile_rows;
}
__host__ __device__ inline GemmTile segment_tile(int expert, int seg_row0, int padded, int valid, int tile_rows,
                                                 int nt, int j, int first) {
  GemmTile tl;
  tl.expert = expert;
  tl.row0 = seg_row0 + j * tile_rows;
  tl.rows = j == nt - 1 ? padded - j * tile_rows : tile_rows;
  tl.first = first;
  tl.count = nt;
  const int v = valid - j * tile_rows;
  tl.valid = v < 0 ? 0 : (v < tl.rows ? v : tl.rows);
  tl.pad[0] = tl.pad[1] = 0;
  return tl;
}
// One launch: tile list a (when non-null) and b (when both are), one CTA
// each, beside the routed token rows of x_perm (row_mode 1: gathered in
// padded-row order by sorted_route_ids; 2: token by token from the inverse
// map route_pos (padded row of each route, -1 dropped), each token row read
// once; 0: none).  Padding rows are written as zeros.
void launch_tiles_and_rows(const int32_t* block_expert, const int32_t* num_padded,
                           const int32_t* sorted_route_ids, int k, int T, int N, int B, int64_t max_rows,
                           const TileListOut* a, const TileListOut* b, int* status, int row_mode,
                           const uint16_t* h, const int32_t* route_pos, int H, uint16_t* x_perm,
                           cudaStream_t s);

// ---- diagnostics
struct RoutingStats {  // same layout as moe_route_stats
  int32_t max_expert_load, min_expert_load, capacity, dropped_tokens, total_routes, reserved;
  double imbalance_ratio, drop_fraction;
};
void launch_routing_stats(const int32_t* topk_idx, long long R, int N, double capacity_factor,
                          int32_t* load_out, RoutingStats* stats, cudaStream_t s);
void launch_router_margin(const float* logits, int T, int N, int k, double* margin, cudaStream_t s);

// ---- combine (k = route slots per token: top_k, or N for expert choice)
void launch_combine(const uint16_t* h, const float* gates, const uint8_t* route_kept,
                    const int32_t* route_pos, const uint16_t* y_perm, const uint16_t* y_shared,
                    uint16_t* out, int T, int H, int k, int64_t max_rows, cudaStream_t s);

}  // namespace moe
