// C ABI of the batch-invariant MoE layer (include/moe_api.h): argument
// validation, workspace carving, TMA tensor maps and the launch sequence.
#include "moe_api.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "kernels.h"

namespace {

using moe::GemmTile;

constexpr int kMaxDevices = 64;
constexpr uint32_t kKnownDebugFlags = 0x3FFFu;
static_assert(MOE_DEBUG_ROUTER_TC == moe::kPathRouterTc && MOE_DEBUG_ROUTER_CHUNKED == moe::kPathRouterChunked &&
                  MOE_DEBUG_ROW_GATHER == moe::kPathRowGather && MOE_DEBUG_ROW_SCATTER == moe::kPathRowScatter &&
                  MOE_DEBUG_NO_DECODE_FRONT == moe::kPathNoDecodeFront &&
                  MOE_DEBUG_REROUTE_SEQUENTIAL == moe::kPathRerouteSequential &&
                  MOE_DEBUG_REROUTE_GRID == moe::kPathRerouteGrid &&
                  MOE_DEBUG_REROUTE_ONE_CTA == moe::kPathRerouteOneCta &&
                  MOE_DEBUG_ROUTER_TILE128 == moe::kPathRouterTile128 &&
                  MOE_DEBUG_ROUTER_TILE64 == moe::kPathRouterTile64,
              "debug flags mirror the internal path flags");
static_assert(MOE_DEV_NOTE_REROUTE_FALLBACK == moe::kDevNoteRerouteFallback, "status bits");

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ----------------------------------------------------------------- config
moe_status check_cfg(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->hidden <= 0 || c->num_experts <= 0 || c->top_k <= 0 || c->intermediate <= 0 ||
      c->block_size <= 0 || c->shared_intermediate < 0 || std::isnan(c->capacity_factor))
    return MOE_ERR_INVALID_ARG;
  if (c->hidden % 128 || c->hidden > 32768) return MOE_ERR_UNSUPPORTED;
  if (c->intermediate % 128 || c->intermediate > 65536) return MOE_ERR_UNSUPPORTED;
  if (c->shared_intermediate % 128 || c->shared_intermediate > 65536) return MOE_ERR_UNSUPPORTED;
  if (c->num_experts > 256) return MOE_ERR_UNSUPPORTED;
  if (c->top_k > c->num_experts || c->top_k > 16) return MOE_ERR_UNSUPPORTED;
  if (c->block_size % 8 || c->block_size > 128 || 128 % c->block_size) return MOE_ERR_UNSUPPORTED;
  if (c->overflow_policy != MOE_OVERFLOW_DROP && c->overflow_policy != MOE_OVERFLOW_REROUTE)
    return MOE_ERR_INVALID_ARG;
  if (c->routing != MOE_ROUTING_TOKEN_CHOICE && c->routing != MOE_ROUTING_EXPERT_CHOICE)
    return MOE_ERR_INVALID_ARG;
  // debug fields: known bits only, no contradictory pair
  const uint32_t f = c->debug_flags;
  if (f & ~kKnownDebugFlags) return MOE_ERR_INVALID_ARG;
  auto both = [f](uint32_t a, uint32_t b) { return (f & a) && (f & b); };
  if (both(MOE_DEBUG_ROUTER_TC, MOE_DEBUG_ROUTER_CHUNKED) || both(MOE_DEBUG_ROW_GATHER, MOE_DEBUG_ROW_SCATTER) ||
      both(MOE_DEBUG_REROUTE_GRID, MOE_DEBUG_REROUTE_ONE_CTA) ||
      both(MOE_DEBUG_ROUTER_TILE128, MOE_DEBUG_ROUTER_TILE64))
    return MOE_ERR_INVALID_ARG;
  if (c->debug_grid_ctas < 0 || c->debug_wait_ns < 0) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe::PathOpts opts_of(const moe_config* c) {
  moe::PathOpts o;
  o.flags = c->debug_flags;
  o.grid_ctas = c->debug_grid_ctas;
  o.wait_ns = (uint64_t)c->debug_wait_ns;
  return o;
}

bool expert_choice(const moe_config* c) { return c->routing == MOE_ROUTING_EXPERT_CHOICE; }

// Route slots per token: k (token choice) or N (expert choice, slot e = expert e).
int slots_of(const moe_config* c) { return expert_choice(c) ? c->num_experts : c->top_k; }

moe_status check_T(const moe_config* c, int32_t T) {
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T > (1 << 20) || (int64_t)T * slots_of(c) >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// Token choice: ceil(cf*T*k/N) or -1 (no limit).  Expert choice: tokens per
// expert, min(ceil(cf*T*k/N), T) with cf = 1 when unset.
int32_t capacity_of(const moe_config* c, int32_t T) {
  if (expert_choice(c)) {
    const double cf = c->capacity_factor > 0.0 ? c->capacity_factor : 1.0;
    const double v = std::ceil(cf * (double)T * (double)c->top_k / (double)c->num_experts);
    return v >= (double)T ? T : (int32_t)v;
  }
  if (!(c->capacity_factor > 0.0)) return -1;
  return (int32_t)std::ceil(c->capacity_factor * (double)T * (double)c->top_k /
                            (double)c->num_experts);
}

bool reroute_active(const moe_config* c, int32_t T) {
  return !expert_choice(c) && c->overflow_policy == MOE_OVERFLOW_REROUTE && capacity_of(c, T) >= 0;
}

// Expert choice: every expert takes exactly C tokens, segment P = C rounded up to B.
int64_t ec_segment_rows(const moe_config* c, int32_t T) {
  const int64_t C = capacity_of(c, T);
  return (C + c->block_size - 1) / c->block_size * c->block_size;
}

int64_t max_rows_of(const moe_config* c, int32_t T) {
  if (expert_choice(c)) return (int64_t)c->num_experts * ec_segment_rows(c, T);
  return (int64_t)T * c->top_k + (int64_t)c->num_experts * (c->block_size - 1);
}
int64_t max_blocks_of(const moe_config* c, int32_t T) {
  if (expert_choice(c)) return max_rows_of(c, T) / c->block_size;
  return (int64_t)T * c->top_k / c->block_size + c->num_experts;
}
int64_t max_gemm_tiles_of(const moe_config* c, int32_t T, int tile_rows) {
  return (max_rows_of(c, T) + tile_rows - 1) / tile_rows + c->num_experts;
}

// ----------------------------------------------------------------- workspace
// Regions, each 256-byte aligned; the status word is always at offset 0.
struct Layout {
  size_t status, logits, wgT, norm_w, rpart, topk, gates, kept, pos, rank, tile_count, seg_off, sorted, blocks,
      num_padded, counts, dropped, route_expert, rerouted, rr_list, rr_hold, rr_cand, rr_ptr, rr_first,
      rr_prefs,
      rr_acc, rr_worst, rr_flag, rr_count, rr_gsync, rr_lcount, rr_lrank, ec_keys, gemm_tiles, num_gemm_tiles,
      gemm_tiles2, num_gemm_tiles2, x_perm, a, y, a_sh, y_sh, h_stage, out_stage, total;
};

Layout layout_of(const moe_config* c, int32_t T) {
  const size_t R = (size_t)T * slots_of(c), N = c->num_experts, H = c->hidden;
  const size_t rows = (size_t)max_rows_of(c, T);
  const size_t dtiles = (R + moe::kDispatchTile - 1) / moe::kDispatchTile;
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, 256);
    return at;
  };
  L.status = take(sizeof(int32_t));
  L.logits = take(sizeof(float) * T * N);
  L.wgT = take(sizeof(uint16_t) * N * H);
  L.norm_w = take(sizeof(float) * N);
  L.rpart = take(sizeof(float) * std::max(moe::chunked_router_part_floats(T, (int)H, (int)N),
                                          moe::route_certified_scratch_floats(T, (int)H)));
  L.topk = take(sizeof(int32_t) * R);
  L.gates = take(sizeof(float) * R);
  L.kept = take(R);
  L.pos = take(sizeof(int32_t) * R);
  L.rank = take(sizeof(int32_t) * R);
  L.tile_count = take(sizeof(int32_t) * dtiles * N);
  L.seg_off = take(sizeof(int32_t) * N);
  L.sorted = take(sizeof(int32_t) * rows);
  L.blocks = take(sizeof(int32_t) * (size_t)max_blocks_of(c, T));
  L.num_padded = take(sizeof(int32_t));
  L.counts = take(sizeof(int32_t) * N);
  L.dropped = take(sizeof(int32_t));
  const bool rr = c->overflow_policy == MOE_OVERFLOW_REROUTE && !expert_choice(c);
  L.route_expert = take(rr ? sizeof(int32_t) * R : 0);
  L.rerouted = take(sizeof(int32_t));
  L.rr_list = take(rr ? sizeof(int32_t) * R : 0);
  L.rr_hold = take(rr ? sizeof(int32_t) * R : 0);
  L.rr_cand = take(rr ? sizeof(int32_t) * R : 0);
  L.rr_ptr = take(rr ? sizeof(int32_t) * R : 0);
  L.rr_first = take(rr ? sizeof(int32_t) * R : 0);
  L.rr_prefs = take(rr ? (size_t)T * moe::kRerouteListLen : 0);
  L.rr_acc = take(sizeof(int32_t) * N);
  L.rr_worst = take(sizeof(int32_t) * N);
  L.rr_flag = take(sizeof(int32_t));
  L.rr_count = take(sizeof(int32_t));
  // the grid-wide rounds use at most R / 1009 + 1 CTAs (chunks of >= 1009 routes)
  const size_t rr_ctas = R / 1000 + 2;
  L.rr_gsync = take(4 * sizeof(uint32_t));
  L.rr_lcount = take(rr ? sizeof(int32_t) * 2 * moe::reroute_exchange_ints((int)rr_ctas, (int)N) : 0);
  L.rr_lrank = take(rr ? sizeof(int32_t) * 2 * R : 0);
  L.ec_keys = take(expert_choice(c) ? sizeof(unsigned long long) * N * T : 0);
  // tile lists of the W13 (128-row) and W2 (256-row) GEMMs
  L.gemm_tiles = take(sizeof(GemmTile) * (size_t)max_gemm_tiles_of(c, T, moe::kW13TileRows));
  L.num_gemm_tiles = take(2 * sizeof(int32_t));   // the tile count, then the GEMM's tile counter
  L.gemm_tiles2 = take(sizeof(GemmTile) * (size_t)max_gemm_tiles_of(c, T, moe::kW2TileRows));
  L.num_gemm_tiles2 = take(2 * sizeof(int32_t));
  // x_perm and a keep one tile of rows of slack so every tile load stays inside them
  L.x_perm = take(sizeof(uint16_t) * (rows + moe::kMaxTileRows) * H);
  L.a = take(sizeof(uint16_t) * (rows + moe::kMaxTileRows) * c->intermediate);
  L.y = take(sizeof(uint16_t) * rows * H);
  const size_t Is = c->shared_intermediate;
  L.a_sh = take(Is ? sizeof(uint16_t) * ((size_t)T + moe::kMaxTileRows) * Is : 0);
  L.y_sh = take(Is ? sizeof(uint16_t) * (size_t)T * H : 0);
  L.h_stage = take(sizeof(uint16_t) * (size_t)T * H);
  L.out_stage = take(sizeof(uint16_t) * (size_t)T * H);
  L.total = off;
  return L;
}

template <class P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

// The routed GEMMs of a forward: which kernel runs each, and the tile list
// each consumes (list a: W13, list b: W2).  A property of the layer's shape,
// except the wide W2 items, which also need enough touched experts.
struct GemmPlan {
  bool pair13, pair2, wide2;
  int rows13, rows2;     // token rows per tile of lists a and b
};

moe_status check_ws(const moe_config* c, int32_t T, const void* ws, size_t ws_bytes);
GemmPlan plan_of(const moe_config* c, int32_t T, int sms);
int num_sms();

// The W13 (a) and W2 (b) tile lists of a forward, in the workspace.
moe::TileListOut list_a(const moe_config* c, int32_t T, const Layout& L, void* ws) {
  const GemmPlan gp = plan_of(c, T, num_sms());
  return moe::TileListOut{at<GemmTile>(ws, L.gemm_tiles), at<int32_t>(ws, L.num_gemm_tiles), gp.rows13,
                          (int)max_gemm_tiles_of(c, T, gp.rows13), at<int32_t>(ws, L.num_gemm_tiles) + 1};
}
moe::TileListOut list_b(const moe_config* c, int32_t T, const Layout& L, void* ws) {
  const GemmPlan gp = plan_of(c, T, num_sms());
  return moe::TileListOut{at<GemmTile>(ws, L.gemm_tiles2), at<int32_t>(ws, L.num_gemm_tiles2), gp.rows2,
                          (int)max_gemm_tiles_of(c, T, gp.rows2), at<int32_t>(ws, L.num_gemm_tiles2) + 1};
}

moe_status check_ws(const moe_config* c, int32_t T, const void* ws, size_t ws_bytes) {
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < layout_of(c, T).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

// ----------------------------------------------------------------- device info / TMA maps
int num_sms() {
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= kMaxDevices) return 0;
  if (!cache[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n;
  }
  return cache[dev];
}

GemmPlan plan_of(const moe_config* c, int32_t T, int sms) {
  const int N = c->num_experts, H = c->hidden, I = c->intermediate;
  const int k = expert_choice(c) ? N : c->top_k;
  GemmPlan p{};
  p.pair13 = moe::gemm_pair_ok(true, I, H) && !(c->debug_flags & MOE_DEBUG_W13_SINGLE);
  p.pair2 = moe::gemm_pair_ok(false, H, I);
  const bool wide_shape = moe::gemm_wide_ok(H, I) ||
                          ((c->debug_flags & MOE_DEBUG_W2_WIDE) && H % moe::kPairFeatW2Wide == 0);
  // wide W2 items (two 256-feature groups per token tile, the same MMAs)
  // where the layer has a long reduction and the batch touches enough
  // experts to keep a quarter of the SMs busy with them (at T = 1 the
  // Mixtral-like W2 took 0.196 ms with them against 0.167 without)
  const long long touched = std::min<long long>(N, (long long)T * k);
  p.wide2 = p.pair2 && wide_shape && touched * (H / moe::kPairFeatW2Wide) * 4 >= sms;
  p.rows13 = p.pair13 ? moe::kPairTileRows : moe::kW13TileRows;
  p.rows2 = moe::kW2TileRows;
  return p;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 2-D map with 128-byte swizzle: `inner` contiguous elements per row,
// `outer` rows, box box_inner x box_outer.
bool map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
            uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn || inner == 0 || outer == 0) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token-tile maps of a GEMM whose tiles have `bn` rows: the full box and the
// 32-row box used for tiles of at most 32 rows.
bool token_maps(CUtensorMap* full, CUtensorMap* small, const void* base, uint64_t inner, uint64_t outer,
                int bn) {
  return map_2d(full, base, inner, outer, 64, (uint32_t)bn) && map_2d(small, base, inner, outer, 64, 32u);
}

moe_status last_cuda() { return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// ----------------------------------------------------------------- stages
bool use_tc_router(const moe_config* c) {
  return c->num_experts % moe::kTileFeat == 0 && moe::route_certified_ok(c->hidden);
}

// Tensor-core logits l_tc = h . W_g (no bias) into `logits` [T, N]: the
// grouped GEMM kernel in identity mode with W_g [H, N] as the weights operand.
moe_status tc_logits(const moe_config* c, int32_t T, const uint16_t* h, const uint16_t* wg,
                     float* logits, void* ws, cudaStream_t s) {
  const Layout L = layout_of(c, T);
  const int H = c->hidden, N = c->num_experts;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  // 64-row token tiles while 128-row ones would not give every SM a tile
  const long long wide_units = (long long)((T + moe::kRouterTileRows - 1) / moe::kRouterTileRows) *
                               (N / moe::kTileFeat);
  int rows = wide_units < sms ? moe::kRouterTileRowsNarrow : moe::kRouterTileRows;
  if (c->debug_flags & MOE_DEBUG_ROUTER_TILE128) rows = moe::kRouterTileRows;
  if (c->debug_flags & MOE_DEBUG_ROUTER_TILE64) rows = moe::kRouterTileRowsNarrow;
  CUtensorMap m_wg, m_h, m_hs;
  if (!map_2d(&m_wg, wg, (uint64_t)N, (uint64_t)H, 64, 64) ||
      !map_2d(&m_h, h, (uint64_t)H, (uint64_t)T, 64, (uint32_t)rows) ||
      !map_2d(&m_hs, h, (uint64_t)H, (uint64_t)T, 64, 32))
    return MOE_ERR_CUDA;
  moe::GemmArgs g{};
  g.K = H;
  g.n_feat_tiles = N / moe::kTileFeat;
  g.w_rows_per_e = H;
  g.identity_T = T;
  g.out = logits;
  g.out_ld = N;
  g.status = at<int>(ws, L.status);
  g.wait_ns = (unsigned long long)c->debug_wait_ns;
  moe::launch_router_gemm(m_wg, m_h, m_hs, g, (T + rows - 1) / rows, sms, s, rows);
  return last_cuda();
}

moe_status route_impl(const moe_config* c, int32_t T, const uint16_t* h, const uint16_t* wg,
                      const float* bias, int32_t* idx, float* gates, float* logits, bool canonical_logits,
                      void* ws, cudaStream_t s, int32_t* n_cand = nullptr) {
  const int H = c->hidden, N = c->num_experts, k = c->top_k;
  if (moe::chunked_router_ok(T, H, N, use_tc_router(c) && !canonical_logits, c->debug_flags) && !n_cand) {
    // a few tokens, or a small W_g: chunk sums spread over many CTAs, the
    // same bits as either path below
    const Layout L = layout_of(c, T);
    moe::launch_router_chunked(h, wg, bias, at<float>(ws, L.rpart), logits, idx, gates, T, H, N, k, s);
    return last_cuda();
  }
  // the certified tensor-core path pays off on batches (same bits as the
  // CUDA-core path)
  if (!canonical_logits && use_tc_router(c) && moe::gemm_smem_ok()) {
    const Layout L = layout_of(c, T);
    uint16_t* wgT = at<uint16_t>(ws, L.wgT);
    float* norm_w = at<float>(ws, L.norm_w);
    moe::launch_gate_prep(wg, wgT, norm_w, H, N, s);
    const moe_status st = tc_logits(c, T, h, wg, logits, ws, s);
    if (st != MOE_OK) return st;
    moe::launch_route_certified(logits, bias, h, wgT, norm_w, T, H, N, k, idx, gates, n_cand,
                                at<float>(ws, L.rpart), s);
    return last_cuda();
  }
  // the tensor-core path is unavailable: the chunked router serves any batch
  const Layout L = layout_of(c, T);
  moe::launch_router_chunked(h, wg, bias, at<float>(ws, L.rpart), logits, idx, gates, T, H, N, k, s);
  return last_cuda();
}

moe_status dispatch_impl(const moe_config* c, int32_t T, const int32_t* idx, uint8_t* kept,
                         int32_t* pos, int32_t* sorted, int32_t* blocks, int32_t* num_padded,
                         int32_t* counts, int32_t* dropped, void* ws, cudaStream_t s) {
  const Layout L = layout_of(c, T);
  moe::launch_dispatch(idx, T, c->num_experts, c->top_k, c->block_size, capacity_of(c, T), kept, pos,
                       sorted, blocks, num_padded, counts, dropped, at<int32_t>(ws, L.rank),
                       at<int32_t>(ws, L.tile_count), at<int32_t>(ws, L.seg_off), at<int>(ws, L.status), s);
  return last_cuda();
}

moe_status reroute_impl(const moe_config* c, int32_t T, const int32_t* idx, const float* logits,
                        uint8_t* kept, int32_t* route_expert, int32_t* pos, int32_t* sorted,
                        int32_t* blocks, int32_t* num_padded, int32_t* counts, int32_t* dropped,
                        int32_t* rerouted, void* ws, cudaStream_t s) {
  // the reroute scratch is laid out for the reroute policy whatever cfg says
  moe_config cr = *c;
  cr.overflow_policy = MOE_OVERFLOW_REROUTE;
  const Layout L = layout_of(&cr, T);
  moe::RerouteScratch sc{at<int32_t>(ws, L.rr_list), at<int32_t>(ws, L.rr_hold), at<int32_t>(ws, L.rr_cand),
                         at<int32_t>(ws, L.rr_ptr), at<int32_t>(ws, L.rr_first), at<uint8_t>(ws, L.rr_prefs),
                         at<int32_t>(ws, L.rr_acc),
                         at<int32_t>(ws, L.rr_worst), at<int32_t>(ws, L.rr_flag),
                         at<int32_t>(ws, L.rr_count), at<uint32_t>(ws, L.rr_gsync),
                         at<int32_t>(ws, L.rr_lcount), at<int32_t>(ws, L.rr_lrank)};
  moe::launch_dispatch_reroute(idx, logits, T, c->num_experts, c->top_k, c->block_size, capacity_of(c, T),
                               kept, route_expert, pos, sorted, blocks, num_padded, counts, dropped,
                               rerouted, at<int32_t>(ws, L.rank), at<int32_t>(ws, L.tile_count),
                               at<int32_t>(ws, L.seg_off), sc, at<int>(ws, L.status), opts_of(c), s);
  return last_cuda();
}

moe_status expert_choice_impl(const moe_config* c, int32_t T, const float* logits, float* gates,
                              uint8_t* kept, int32_t* pos, int32_t* sorted, int32_t* blocks,
                              int32_t* num_padded, int32_t* counts, void* ws, cudaStream_t s) {
  const Layout L = layout_of(c, T);
  moe::launch_expert_choice(logits, T, c->num_experts, capacity_of(c, T), c->block_size,
                            at<unsigned long long>(ws, L.ec_keys), gates, kept, pos, sorted, blocks,
                            num_padded, counts, s);
  return last_cuda();
}

// x_perm token by token (each h row read once) when h exceeds 48 MB: the
// segment-order gather fetches a row once per slot, from DRAM when h does
// not stay in L2 (measured on the DeepSeek-like layer, whose row copy shares
// the SMs with the shared expert: 4.488 -> 4.452 ms at T = 4096, 11.92 ->
// 11.87 ms at T = 16448; no change at 33 MB).  The caller's path flags may
// force one (both write the same rows).
bool scatter_rows_ok(int T, int H, uint32_t path_flags) {
  if (path_flags & MOE_DEBUG_ROW_GATHER) return false;
  if (path_flags & MOE_DEBUG_ROW_SCATTER) return true;
  return (long long)T * H * 2 > (48ll << 20);
}

struct Marks;
moe_status ffn_impl(const moe_config* c, int32_t T, const uint16_t* h, const uint16_t* w13,
                    const uint16_t* w2, const uint16_t* w13s, const uint16_t* w2s, const int32_t* sorted,
                    const int32_t* blocks, const int32_t* num_padded, uint16_t* y_perm, uint16_t* y_shared,
                    void* ws, cudaStream_t s, const Marks* mk = nullptr, bool tiles_ready = false,
                    bool skip_shared = false, const int32_t* route_pos = nullptr, bool rows_ready = false);
void mark(const Marks* mk, int i);

// The shared expert (identity mode over h; every token, no routing): W13 then
// W2 into y_shared.  It depends on h alone, so the forward runs it on a
// second stream alongside routing, dispatch and the routed GEMMs.
moe_status shared_ffn_impl(const moe_config* c, int32_t T, const uint16_t* h, const uint16_t* w13s,
                           const uint16_t* w2s, uint16_t* y_shared, void* ws, cudaStream_t s) {
  const Layout L = layout_of(c, T);
  const int H = c->hidden, Is = c->shared_intermediate;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  int* status = at<int>(ws, L.status);
  const bool pair2 = moe::gemm_pair_ok(false, H, Is);
  const int box2 = pair2 ? moe::kPairBoxRows : moe::kW2TileRows;
  uint16_t* ash = at<uint16_t>(ws, L.a_sh);
  const bool spair13 = moe::gemm_pair_ok(true, Is, H);
  const int sbox13 = spair13 ? moe::kPairBoxRows : moe::kW13TileRows;
  const int srows13 = spair13 ? moe::kPairTileRows : moe::kW13TileRows;
  CUtensorMap m_w13s, m_w2s, m_ash, m_ashs, m_h, m_hs;
  // the last tile of h may run past row T-1: TMA fills those rows with zeros
  if (!token_maps(&m_h, &m_hs, h, (uint64_t)H, (uint64_t)T, sbox13) ||
      !map_2d(&m_w13s, w13s, 2ull * Is, (uint64_t)H, 64, 64) ||
      !map_2d(&m_w2s, w2s, (uint64_t)H, (uint64_t)Is, 64, 64) ||
      !token_maps(&m_ash, &m_ashs, ash, (uint64_t)Is, (uint64_t)T + moe::kMaxTileRows, box2))
    return MOE_ERR_CUDA;
  moe::GemmArgs s13{};
  s13.K = H;
  s13.n_feat_tiles = spair13 ? Is / moe::kPairFeatW13 : Is / moe::kTileFeat;
  s13.w_rows_per_e = H;
  s13.up_col = Is;
  s13.identity_T = T;
  s13.out = ash;
  s13.out_ld = Is;
  s13.status = status;
  s13.pair = spair13 ? 1 : 0;
  s13.decode = T <= moe::kDecodeMaxT ? 1 : 0;   // identity tiles of at most T rows
  s13.wait_ns = (unsigned long long)c->debug_wait_ns;
  moe::launch_w13_gemm(m_w13s, m_h, m_hs, s13, (T + srows13 - 1) / srows13, sms, s);
  moe::GemmArgs s2 = s13;
  s2.K = Is;
  s2.n_feat_tiles = pair2 ? H / moe::kPairFeatW2 : H / moe::kTileFeat;
  s2.w_rows_per_e = Is;
  s2.up_col = 0;
  s2.out = y_shared;
  s2.out_ld = H;
  s2.out_bf16 = 1;
  s2.pair = pair2 ? 1 : 0;
  s2.decode = T <= moe::kDecodeMaxT ? 1 : 0;
  moe::launch_w2_gemm(m_w2s, m_ash, m_ashs, s2, (T + moe::kW2TileRows - 1) / moe::kW2TileRows, sms, s);
  return last_cuda();
}

moe_status ffn_impl(const moe_config* c, int32_t T, const uint16_t* h, const uint16_t* w13,
                    const uint16_t* w2, const uint16_t* w13s, const uint16_t* w2s, const int32_t* sorted,
                    const int32_t* blocks, const int32_t* num_padded, uint16_t* y_perm, uint16_t* y_shared,
                    void* ws, cudaStream_t s, const Marks* mk, bool tiles_ready, bool skip_shared,
                    const int32_t* route_pos, bool rows_ready) {
  const Layout L = layout_of(c, T);
  const int N = c->num_experts, H = c->hidden, I = c->intermediate, k = slots_of(c);
  const int64_t rows = max_rows_of(c, T);
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  const GemmPlan gp = plan_of(c, T, sms);
  const int max_tiles13 = (int)max_gemm_tiles_of(c, T, gp.rows13);
  const int max_tiles2 = (int)max_gemm_tiles_of(c, T, gp.rows2);
  int* status = at<int>(ws, L.status);
  GemmTile* tiles13 = at<GemmTile>(ws, L.gemm_tiles);
  int32_t* ntiles13 = at<int32_t>(ws, L.num_gemm_tiles);
  GemmTile* tiles2 = at<GemmTile>(ws, L.gemm_tiles2);
  int32_t* ntiles2 = at<int32_t>(ws, L.num_gemm_tiles2);
  uint16_t* a = at<uint16_t>(ws, L.a);
  uint16_t* x_perm = at<uint16_t>(ws, L.x_perm);

  {
    // the tile lists (unless the small-batch dispatch built both) and the
    // routed rows (unless the decode front copied them), in one launch
    const moe::TileListOut l13{tiles13, ntiles13, gp.rows13, max_tiles13, ntiles13 + 1};
    const moe::TileListOut l2{tiles2, ntiles2, gp.rows2, max_tiles2, ntiles2 + 1};
    const int row_mode = rows_ready ? 0 : (route_pos && scatter_rows_ok(T, H, c->debug_flags) ? 2 : 1);
    moe::launch_tiles_and_rows(blocks, num_padded, sorted, k, T, N, c->block_size, rows,
                               tiles_ready ? nullptr : &l13, tiles_ready ? nullptr : &l2, status, row_mode, h,
                               route_pos, H, x_perm, s);
  }
  mark(mk, 3);

  // CTA-pair kernels where the output features are a multiple of 256 (a
  // property of the layer, the same for every T); they take the 256-row tile
  // list and load 128-row token boxes per CTA
  const bool pair13 = gp.pair13, pair2 = gp.pair2;
  const int box13 = pair13 ? moe::kPairBoxRows : moe::kW13TileRows;
  const int box2 = pair2 ? moe::kPairBoxRows : moe::kW2TileRows;
  CUtensorMap m_w13, m_x, m_xs, m_w2, m_a, m_as;
  if (!map_2d(&m_w13, w13, 2ull * I, (uint64_t)N * H, 64, 64) ||
      !token_maps(&m_x, &m_xs, x_perm, (uint64_t)H, (uint64_t)(rows + moe::kMaxTileRows), box13) ||
      !map_2d(&m_w2, w2, (uint64_t)H, (uint64_t)N * I, 64, 64) ||
      !token_maps(&m_a, &m_as, a, (uint64_t)I, (uint64_t)(rows + moe::kMaxTileRows), box2))
    return MOE_ERR_CUDA;

  moe::GemmArgs g13{};
  g13.K = H;
  g13.n_feat_tiles = pair13 ? I / moe::kPairFeatW13 : I / moe::kTileFeat;
  g13.w_rows_per_e = H;
  g13.up_col = I;
  g13.tiles = tiles13;
  g13.num_tiles = ntiles13;
  // the one-CTA kernel takes its tiles from a counter (zeroed with the tile
  // count): whichever CTA is free takes the next tile.  The pair kernels
  // keep the fixed assignment (item u + n * pairs), which measured faster.
  g13.next_item = pair13 ? nullptr : ntiles13 + 1;
  g13.identity_T = 0;
  g13.out = a;
  g13.out_ld = I;
  g13.status = status;
  g13.pair = pair13 ? 1 : 0;
  // decode instances: no tile of this call holds more than kDecodeMaxT
  // routed rows — at most that many tokens in the forward (a token routes to
  // an expert at most once), or that many routes in all for a caller's own
  // block list
  const bool decode =
      T <= moe::kDecodeMaxT && (route_pos != nullptr || (long long)T * k <= moe::kDecodeMaxT);
  g13.decode = decode ? 1 : 0;
  g13.wait_ns = (unsigned long long)c->debug_wait_ns;
  moe::launch_w13_gemm(m_w13, m_x, m_xs, g13, max_tiles13, sms, s);
  mark(mk, 4);

  const bool wide2 = gp.wide2;
  moe::GemmArgs g2 = g13;
  g2.K = I;
  g2.n_feat_tiles = wide2 ? H / moe::kPairFeatW2Wide : (pair2 ? H / moe::kPairFeatW2 : H / moe::kTileFeat);
  g2.w_rows_per_e = I;
  g2.up_col = 0;
  g2.tiles = tiles2;
  g2.num_tiles = ntiles2;
  g2.next_item = pair2 ? nullptr : ntiles2 + 1;
  g2.out = y_perm;
  g2.out_ld = H;
  g2.out_bf16 = 1;
  g2.pair = pair2 ? 1 : 0;
  g2.wide = wide2 ? 1 : 0;
  g2.decode = (decode && !wide2) ? 1 : 0;
  moe::launch_w2_gemm(m_w2, m_a, m_as, g2, max_tiles2, sms, s);
  mark(mk, 5);

  if (!skip_shared && c->shared_intermediate > 0) {
    const moe_status st = shared_ffn_impl(c, T, h, w13s, w2s, y_shared, ws, s);
    if (st != MOE_OK) return st;
  }
  return last_cuda();
}

// Records events[i] on s if events are given (stage boundary i).
struct Marks {
  void* const* ev;
  cudaStream_t s;
  void at(int i) const {
    if (ev) cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), s);
  }
};

void mark(const Marks* mk, int i) {
  if (mk) mk->at(i);
}

// Second stream of a device for the shared expert, with the fork and join
// events.  One forward at a time enqueues on it (the events are reused).
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

std::mutex& side_mutex() {
  static std::mutex m;
  return m;
}

// Called with side_mutex() held.
bool side_stream(SideStream* out) {
  static SideStream cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  SideStream& c = cache[dev];
  if (!c.stream) {
    if (cudaStreamCreateWithFlags(&c.stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&c.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c.join, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      c = SideStream{};
      return false;
    }
  }
  *out = c;
  return true;
}

moe_status forward_impl(const moe_config* c, int32_t T, const uint16_t* h, const uint16_t* wg,
                        const float* bias, const uint16_t* w13, const uint16_t* w2, const uint16_t* w13s,
                        const uint16_t* w2s, uint16_t* out, void* ws, cudaStream_t s,
                        void* const* events = nullptr) {
  const Marks mk{events, s};
  const Layout L = layout_of(c, T);
  int32_t* idx = at<int32_t>(ws, L.topk);
  float* gates = at<float>(ws, L.gates);
  uint8_t* kept = at<uint8_t>(ws, L.kept);
  int32_t* pos = at<int32_t>(ws, L.pos);
  int32_t* sorted = at<int32_t>(ws, L.sorted);
  int32_t* blocks = at<int32_t>(ws, L.blocks);
  int32_t* num_padded = at<int32_t>(ws, L.num_padded);
  uint16_t* y = at<uint16_t>(ws, L.y);
  uint16_t* ysh = c->shared_intermediate ? at<uint16_t>(ws, L.y_sh) : nullptr;
  float* logits = at<float>(ws, L.logits);
  int32_t* counts = at<int32_t>(ws, L.counts);
  moe_status st = MOE_OK;
  bool tiles_ready = false, rows_ready = false;
  mk.at(0);
  // the shared expert needs h alone: it runs on a second stream from the end
  // of routing (the router, latency-bound, keeps the SMs to itself) and
  // joins before the combine; it overlaps dispatch, the row gather and the
  // routed GEMMs
  std::unique_lock<std::mutex> side_lock;
  SideStream side;
  // (the debug flag MOE_DEBUG_SHARED_SERIAL runs it on `s` after the routed GEMMs instead)
  const bool shared = c->shared_intermediate > 0 && !(c->debug_flags & MOE_DEBUG_SHARED_SERIAL);
  bool forked = false;
  auto fork_shared = [&]() -> moe_status {
    if (!shared) return MOE_OK;
    side_lock = std::unique_lock<std::mutex>(side_mutex());
    if (!side_stream(&side)) return MOE_ERR_CUDA;
    if (cudaEventRecord(side.fork, s) != cudaSuccess ||
        cudaStreamWaitEvent(side.stream, side.fork, 0) != cudaSuccess)
      return last_cuda();
    forked = true;
    moe_status r = shared_ffn_impl(c, T, h, w13s, w2s, ysh, ws, side.stream);
    if (cudaEventRecord(side.join, side.stream) != cudaSuccess && r == MOE_OK) r = last_cuda();
    return r;
  };
  if (expert_choice(c)) {
    // every logit in the canonical order, then each expert takes its tokens
    moe::launch_router_chunked(h, wg, bias, at<float>(ws, L.rpart), logits, nullptr, nullptr, T, c->hidden,
                               c->num_experts, c->top_k, s);
    mk.at(1);
    st = fork_shared();
    if (st == MOE_OK)
      st = expert_choice_impl(c, T, logits, gates, kept, pos, sorted, blocks, num_padded, counts, ws, s);
  } else if (reroute_active(c, T)) {
    // rerouting ranks every expert of an overflowing token: canonical logits
    st = route_impl(c, T, h, wg, bias, idx, gates, logits, true, ws, s);
    mk.at(1);
    if (st == MOE_OK) st = fork_shared();
    if (st == MOE_OK)
      st = reroute_impl(c, T, idx, logits, kept, at<int32_t>(ws, L.route_expert), pos, sorted, blocks,
                        num_padded, counts, at<int32_t>(ws, L.dropped), at<int32_t>(ws, L.rerouted), ws, s);
  } else if (moe::decode_front_ok(T, c->hidden, c->num_experts, c->top_k, c->debug_flags)) {
    // a few tokens: the router's chunk sums, then routing, dispatch, both
    // tile lists and the routed rows in one more launch (the same bits as
    // the separate kernels)
    moe::launch_decode_front(h, wg, bias, at<float>(ws, L.rpart), T, c->hidden, c->num_experts, c->top_k,
                             c->block_size, capacity_of(c, T),
                             idx, gates, kept, pos, sorted, blocks, num_padded, counts, at<int32_t>(ws, L.dropped),
                             list_a(c, T, L, ws), list_b(c, T, L, ws), at<uint16_t>(ws, L.x_perm),
                             max_rows_of(c, T), at<int>(ws, L.status), s);
    st = last_cuda();
    mk.at(1);
    if (st == MOE_OK) st = fork_shared();
    tiles_ready = true;
    rows_ready = true;
  } else {
    st = route_impl(c, T, h, wg, bias, idx, gates, logits, false, ws, s);
    mk.at(1);
    if (st == MOE_OK) st = fork_shared();
    // (an error is reported below, after the shared-expert branch has joined)
    if (st == MOE_OK && moe::dispatch_small_ok((long long)T * c->top_k)) {
      // a few routes: dispatch, alignment and both tile lists in one launch
      moe::launch_dispatch_small(idx, T * c->top_k, c->num_experts, c->block_size, capacity_of(c, T), kept, pos,
                                 sorted, blocks, num_padded, counts, at<int32_t>(ws, L.dropped),
                                 list_a(c, T, L, ws), list_b(c, T, L, ws),
                                 at<int>(ws, L.status), s);
      tiles_ready = true;
      st = last_cuda();
    } else if (st == MOE_OK) {
      st = dispatch_impl(c, T, idx, kept, pos, sorted, blocks, num_padded, counts, at<int32_t>(ws, L.dropped),
                         ws, s);
    }
  }
  if (st != MOE_OK) {
    if (forked) cudaStreamWaitEvent(s, side.join, 0);   // leave no branch of a capture unjoined
    return st;
  }
  mk.at(2);
  st = ffn_impl(c, T, h, w13, w2, w13s, w2s, sorted, blocks, num_padded, y, ysh, ws, s, &mk, tiles_ready,
                /*skip_shared=*/shared, pos, rows_ready);
  if (forked && cudaStreamWaitEvent(s, side.join, 0) != cudaSuccess && st == MOE_OK) st = last_cuda();
  if (st != MOE_OK) return st;
  mk.at(6);
  moe::launch_combine(h, gates, kept, pos, y, ysh, out, T, c->hidden, slots_of(c), max_rows_of(c, T), s);
  mk.at(7);
  return last_cuda();
}

#define MOE_TRY(x)                   \
  do {                               \
    const moe_status _st = (x);      \
    if (_st != MOE_OK) return _st;   \
  } while (0)

moe_status need(const void* p) { return (p && aligned16(p)) ? MOE_OK : MOE_ERR_INVALID_ARG; }
moe_status opt(const void* p) { return (!p || aligned16(p)) ? MOE_OK : MOE_ERR_INVALID_ARG; }

moe_status check_shared(const moe_config* c, const void* w13s, const void* w2s) {
  if (c->shared_intermediate > 0) {
    MOE_TRY(need(w13s));
    MOE_TRY(need(w2s));
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE: return "device status word set";
  }
  return "unknown status";
}

moe_status moe_check_config(const moe_config* cfg) { return check_cfg(cfg); }

int32_t moe_capacity(const moe_config* cfg, int32_t T) {
  if (check_cfg(cfg) != MOE_OK || T < 0) return -1;
  return capacity_of(cfg, T);
}

int64_t moe_max_padded_rows(const moe_config* cfg, int32_t T) {
  if (check_cfg(cfg) != MOE_OK || T < 0) return 0;
  return max_rows_of(cfg, T);
}

int64_t moe_max_blocks(const moe_config* cfg, int32_t T) {
  if (check_cfg(cfg) != MOE_OK || T < 0) return 0;
  return max_blocks_of(cfg, T);
}

size_t moe_workspace_bytes(const moe_config* cfg, int32_t max_tokens) {
  if (check_cfg(cfg) != MOE_OK || check_T(cfg, max_tokens) != MOE_OK) return 0;
  return layout_of(cfg, max_tokens).total;
}

moe_status moe_route(const moe_config* cfg, int32_t T, const uint16_t* h, const uint16_t* w_gate,
                     const float* router_bias, int32_t* topk_idx, float* topk_gate, float* logits_out,
                     void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_T(cfg, T));
  if (T == 0) return MOE_OK;
  MOE_TRY(need(h));
  MOE_TRY(need(w_gate));
  MOE_TRY(opt(router_bias));
  MOE_TRY(need(topk_idx));
  MOE_TRY(need(topk_gate));
  MOE_TRY(opt(logits_out));
  MOE_TRY(check_ws(cfg, T, ws, ws_bytes));
  // with logits_out the canonical fp32 logits of every expert are produced
  // (CUDA-core router); without, large-N layers use the tensor-core router
  // with the certified filter (same indices and gates, bit for bit)
  float* logits = logits_out ? logits_out : at<float>(ws, layout_of(cfg, T).logits);
  return route_impl(cfg, T, h, w_gate, router_bias, topk_idx, topk_gate, logits, logits_out != nullptr,
                    ws, static_cast<cudaStream_t>(stream));
}

moe_status moe_dispatch_align(const moe_config* cfg, int32_t T, const int32_t* topk_idx,
                              uint8_t* route_kept, int32_t* route_pos, int32_t* sorted_route_ids,
                              int32_t* block_expert, int32_t* num_padded, int32_t* expert_counts,
                              int32_t* num_dropped, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_T(cfg, T));
  if (T == 0) return MOE_OK;
  MOE_TRY(need(topk_idx));
  MOE_TRY(need(route_kept));
  MOE_TRY(need(route_pos));
  MOE_TRY(need(sorted_route_ids));
  MOE_TRY(need(block_expert));
  MOE_TRY(need(num_padded));
  MOE_TRY(need(expert_counts));
  MOE_TRY(need(num_dropped));
  // the drop policy only: never drop routes the configuration asks to keep
  if (expert_choice(cfg) || reroute_active(cfg, T)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(cfg, T, ws, ws_bytes));
  return dispatch_impl(cfg, T, topk_idx, route_kept, route_pos, sorted_route_ids, block_expert,
                       num_padded, expert_counts, num_dropped, ws, static_cast<cudaStream_t>(stream));
}

moe_status moe_dispatch_align_shard(const moe_config* cfg, int32_t T, int32_t global_tokens,
                                    const int32_t* topk_idx, const int32_t* expert_offset,
                                    uint8_t* route_kept, int32_t* route_pos, int32_t* sorted_route_ids,
                                    int32_t* block_expert, int32_t* num_padded, int32_t* expert_counts,
                                    int32_t* num_dropped, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_T(cfg, T));
  if (global_tokens < T) return MOE_ERR_INVALID_ARG;
  if (expert_choice(cfg) || cfg->overflow_policy == MOE_OVERFLOW_REROUTE) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  MOE_TRY(need(topk_idx));
  MOE_TRY(opt(expert_offset));
  MOE_TRY(need(route_kept));
  MOE_TRY(need(route_pos));
  MOE_TRY(need(sorted_route_ids));
  MOE_TRY(need(block_expert));
  MOE_TRY(need(num_padded));
  MOE_TRY(need(expert_counts));
  MOE_TRY(need(num_dropped));
  MOE_TRY(check_ws(cfg, T, ws, ws_bytes));
  const Layout L = layout_of(cfg, T);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  moe::launch_dispatch(topk_idx, T, cfg->num_experts, cfg->top_k, cfg->block_size, capacity_of(cfg, global_tokens),
                       route_kept, route_pos, sorted_route_ids, block_expert, num_padded, expert_counts, num_dropped,
                       at<int32_t>(ws, L.rank), at<int32_t>(ws, L.tile_count), at<int32_t>(ws, L.seg_off),
                       at<int>(ws, L.status), s, expert_offset);
  return last_cuda();
}

moe_status moe_dispatch_align_reroute(const moe_config* cfg, int32_t T, const int32_t* topk_idx,
                                      const float* logits, uint8_t* route_kept, int32_t* route_expert,
                                      int32_t* route_pos, int32_t* sorted_route_ids,
                                      int32_t* block_expert, int32_t* num_padded,
                                      int32_t* expert_counts, int32_t* num_dropped,
                                      int32_t* num_rerouted, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_T(cfg, T));
  if (expert_choice(cfg)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  MOE_TRY(need(topk_idx));
  MOE_TRY(need(logits));
  MOE_TRY(need(route_kept));
  MOE_TRY(need(route_expert));
  MOE_TRY(need(route_pos));
  MOE_TRY(need(sorted_route_ids));
  MOE_TRY(need(block_expert));
  MOE_TRY(need(num_padded));
  MOE_TRY(need(expert_counts));
  MOE_TRY(need(num_dropped));
  MOE_TRY(need(num_rerouted));
  moe_config cr = *cfg;
  cr.overflow_policy = MOE_OVERFLOW_REROUTE;
  MOE_TRY(check_ws(&cr, T, ws, ws_bytes));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (capacity_of(cfg, T) < 0) {
    // no capacity: nothing overflows; every route keeps its expert
    MOE_TRY(dispatch_impl(cfg, T, topk_idx, route_kept, route_pos, sorted_route_ids, block_expert,
                          num_padded, expert_counts, num_dropped, ws, s));
    if (cudaMemcpyAsync(route_expert, topk_idx, sizeof(int32_t) * (size_t)T * cfg->top_k,
                        cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
        cudaMemsetAsync(num_rerouted, 0, sizeof(int32_t), s) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  return reroute_impl(cfg, T, topk_idx, logits, route_kept, route_expert, route_pos, sorted_route_ids,
                      block_expert, num_padded, expert_counts, num_dropped, num_rerouted, ws, s);
}

moe_status moe_route_expert_choice(const moe_config* cfg, int32_t T, const float* logits, float* gates,
                                   uint8_t* route_kept, int32_t* route_pos, int32_t* sorted_route_ids,
                                   int32_t* block_expert, int32_t* num_padded, int32_t* expert_counts,
                                   void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_T(cfg, T));
  if (!expert_choice(cfg)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  MOE_TRY(need(logits));
  MOE_TRY(need(gates));
  MOE_TRY(need(route_kept));
  MOE_TRY(need(route_pos));
  MOE_TRY(need(sorted_route_ids));
  MOE_TRY(need(block_expert));
  MOE_TRY(need(num_padded));
  MOE_TRY(need(expert_counts));
  MOE_TRY(check_ws(cfg, T, ws, ws_bytes));
  return expert_choice_impl(cfg, T, logits, gates, route_kept, route_pos, sorted_route_ids, block_expert,
                            num_padded, expert_counts, ws, static_cast<cudaStream_t>(stream));
}

moe_status moe_router_logits(const moe_config* cfg, int32_t T, const uint16_t* h, const uint16_t* w_gate,
                             const float* router_bias, float* logits_out, void* ws, size_t ws_bytes,
                             void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_T(cfg, T));
  if (T == 0) return MOE_OK;
  MOE_TRY(need(h));
  MOE_TRY(need(w_gate));
  MOE_TRY(opt(router_bias));
  MOE_TRY(need(logits_out));
  MOE_TRY(check_ws(cfg, T, ws, ws_bytes));
  moe::launch_router_chunked(h, w_gate, router_bias, at<float>(ws, layout_of(cfg, T).rpart), logits_out,
                             nullptr, nullptr, T, cfg->hidden, cfg->num_experts, cfg->top_k,
                             static_cast<cudaStream_t>(stream));
  return last_cuda();
}

moe_status moe_routing_stats(const moe_config* cfg, int32_t T, const int32_t* topk_idx,
                             double capacity_factor, int32_t* expert_load, moe_route_stats* stats,
                             void* stream) {
  static_assert(sizeof(moe_route_stats) == sizeof(moe::RoutingStats), "stats layout");
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_T(cfg, T));
  if (std::isnan(capacity_factor) || capacity_factor < 0.0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  MOE_TRY(need(topk_idx));
  MOE_TRY(need(expert_load));
  MOE_TRY(need(stats));
  moe::launch_routing_stats(topk_idx, (long long)T * cfg->top_k, cfg->num_experts, capacity_factor,
                            expert_load, reinterpret_cast<moe::RoutingStats*>(stats),
                            static_cast<cudaStream_t>(stream));
  return last_cuda();
}

moe_status moe_router_margin(const moe_config* cfg, int32_t T, const float* logits, double* margin,
                             void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_T(cfg, T));
  if (T == 0) return MOE_OK;
  MOE_TRY(need(logits));
  MOE_TRY(need(margin));
  moe::launch_router_margin(logits, T, cfg->num_experts, cfg->top_k, margin,
                            static_cast<cudaStream_t>(stream));
  return last_cuda();
}

moe_status moe_expert_ffn(const moe_config* cfg, int32_t T, const uint16_t* h, const uint16_t* w13,
                          const uint16_t* w2, const uint16_t* w13_shared, const uint16_t* w2_shared,
                          const int32_t* sorted_route_ids, const int32_t* block_expert,
                          const int32_t* num_padded, uint16_t* y_perm, uint16_t* y_shared, void* ws,
                          size_t ws_bytes, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_T(cfg, T));
  if (T == 0) return MOE_OK;
  MOE_TRY(need(h));
  MOE_TRY(need(w13));
  MOE_TRY(need(w2));
  MOE_TRY(check_shared(cfg, w13_shared, w2_shared));
  if (cfg->shared_intermediate > 0) MOE_TRY(need(y_shared));
  MOE_TRY(need(sorted_route_ids));
  MOE_TRY(need(block_expert));
  MOE_TRY(need(num_padded));
  MOE_TRY(need(y_perm));
  MOE_TRY(check_ws(cfg, T, ws, ws_bytes));
  if (!moe::gemm_smem_ok()) return MOE_ERR_UNSUPPORTED;
  return ffn_impl(cfg, T, h, w13, w2, w13_shared, w2_shared, sorted_route_ids, block_expert, num_padded,
                  y_perm, cfg->shared_intermediate > 0 ? y_shared : nullptr, ws,
                  static_cast<cudaStream_t>(stream));
}

moe_status moe_combine(const moe_config* cfg, int32_t T, const uint16_t* h, const float* topk_gate,
                       const uint8_t* route_kept, const int32_t* route_pos, const uint16_t* y_perm,
                       const uint16_t* y_shared, uint16_t* out, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_T(cfg, T));
  if (T == 0) return MOE_OK;
  MOE_TRY(need(h));
  MOE_TRY(need(topk_gate));
  MOE_TRY(need(route_kept));
  MOE_TRY(need(route_pos));
  MOE_TRY(need(y_perm));
  MOE_TRY(opt(y_shared));
  MOE_TRY(need(out));
  moe::launch_combine(h, topk_gate, route_kept, route_pos, y_perm, y_shared, out, T, cfg->hidden,
                      slots_of(cfg), max_rows_of(cfg, T), static_cast<cudaStream_t>(stream));
  return last_cuda();
}

moe_status moe_forward(const moe_config* cfg, int32_t T, const uint16_t* h, const uint16_t* w_gate,
                       const float* router_bias, const uint16_t* w13, const uint16_t* w2,
                       const uint16_t* w13_shared, const uint16_t* w2_shared, uint16_t* out, void* ws,
                       size_t ws_bytes, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_T(cfg, T));
  if (T == 0) return MOE_OK;
  MOE_TRY(need(h));
  MOE_TRY(need(w_gate));
  MOE_TRY(opt(router_bias));
  MOE_TRY(need(w13));
  MOE_TRY(need(w2));
  MOE_TRY(check_shared(cfg, w13_shared, w2_shared));
  MOE_TRY(need(out));
  MOE_TRY(check_ws(cfg, T, ws, ws_bytes));
  if (!moe::gemm_smem_ok()) return MOE_ERR_UNSUPPORTED;
  return forward_impl(cfg, T, h, w_gate, router_bias, w13, w2, w13_shared, w2_shared, out, ws,
                      static_cast<cudaStream_t>(stream));
}

moe_status moe_forward_timed(const moe_config* cfg, int32_t T, const uint16_t* h,
                             const uint16_t* w_gate, const float* router_bias, const uint16_t* w13,
                             const uint16_t* w2, const uint16_t* w13_shared, const uint16_t* w2_shared,
                             uint16_t* out, void* ws, size_t ws_bytes, void* const* events,
                             int32_t n_events, void* stream) {
  if (!events || n_events < 8) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 8; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_T(cfg, T));
  if (T == 0) return MOE_OK;
  MOE_TRY(need(h));
  MOE_TRY(need(w_gate));
  MOE_TRY(opt(router_bias));
  MOE_TRY(need(w13));
  MOE_TRY(need(w2));
  MOE_TRY(check_shared(cfg, w13_shared, w2_shared));
  MOE_TRY(need(out));
  MOE_TRY(check_ws(cfg, T, ws, ws_bytes));
  if (!moe::gemm_smem_ok()) return MOE_ERR_UNSUPPORTED;
  return forward_impl(cfg, T, h, w_gate, router_bias, w13, w2, w13_shared, w2_shared, out, ws,
                      static_cast<cudaStream_t>(stream), events);
}

int32_t moe_forward_launch_count(const moe_config* cfg, int32_t T) {
  if (check_cfg(cfg) != MOE_OK || T < 0) return 0;
  if (T == 0) return 0;
  // router + dispatch, then the tile lists with the routed-row copy 1 (one
  // launch; the row copy alone after the small-batch dispatch, nothing after
  // the decode front) + W13 + W2 + combine 1 (+ shared W13, W2).  Router:
  // chunk sums + reduce/top-k = 2 (chunked router), or on the tensor cores
  // W_g preparation, GEMM, candidate filter, tiled recompute, finalize = 5.
  // Dispatch: count, scan, scatter = 3, or for at most 1024 routes one
  // launch that also builds both tile lists; with reroute count, scan,
  // preference lists, deferred acceptance, check, sequential fallback
  // (returns at once unless the check failed), count, scan, scatter = 9
  // after the CUDA-core router.  Expert choice: logits (2 launches), scores,
  // selection.  At most two tokens: chunk sums, then one launch for the
  // reduce, top-k, dispatch, tile lists and row gather.
  const bool chunked =
      moe::chunked_router_ok(T, cfg->hidden, cfg->num_experts, use_tc_router(cfg), cfg->debug_flags);
  const int router = chunked ? 2 : (use_tc_router(cfg) ? 5 : 2);
  int front = 0, rows = 1;
  if (expert_choice(cfg)) {   // logits (chunked router, 2), scores, selection
    front = 2 + 2;
  } else if (cfg->overflow_policy == MOE_OVERFLOW_REROUTE && cfg->capacity_factor > 0.0) {
    front = 2 + 9;
  } else if (moe::decode_front_ok(T, cfg->hidden, cfg->num_experts, cfg->top_k, cfg->debug_flags)) {
    // chunk sums, then routing, dispatch, tile lists and the routed rows
    front = 2;
    rows = 0;
  } else if (moe::dispatch_small_ok((long long)T * cfg->top_k)) {
    // dispatch and both tile lists in one launch
    front = router + 1;
  } else {
    front = router + 3;
  }
  return front + rows + 2 + 1 + (cfg->shared_intermediate > 0 ? 2 : 0);
}

moe_status moe_router_tc_logits(const moe_config* cfg, int32_t T, const uint16_t* h,
                                const uint16_t* w_gate, float* logits_out, void* ws, size_t ws_bytes,
                                void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_T(cfg, T));
  if (T == 0) return MOE_OK;
  if (!use_tc_router(cfg)) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(need(h));
  MOE_TRY(need(w_gate));
  MOE_TRY(need(logits_out));
  MOE_TRY(check_ws(cfg, T, ws, ws_bytes));
  if (!moe::gemm_smem_ok()) return MOE_ERR_UNSUPPORTED;
  return tc_logits(cfg, T, h, w_gate, logits_out, ws, static_cast<cudaStream_t>(stream));
}

moe_status moe_route_filtered(const moe_config* cfg, int32_t T, const uint16_t* h,
                              const uint16_t* w_gate, const float* router_bias, int32_t* topk_idx,
                              float* topk_gate, int32_t* n_candidates, void* ws, size_t ws_bytes,
                              void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_T(cfg, T));
  if (T == 0) return MOE_OK;
  if (!use_tc_router(cfg) || !moe::gemm_smem_ok()) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(need(h));
  MOE_TRY(need(w_gate));
  MOE_TRY(opt(router_bias));
  MOE_TRY(need(topk_idx));
  MOE_TRY(need(topk_gate));
  MOE_TRY(need(n_candidates));
  MOE_TRY(check_ws(cfg, T, ws, ws_bytes));
  return route_impl(cfg, T, h, w_gate, router_bias, topk_idx, topk_gate,
                    at<float>(ws, layout_of(cfg, T).logits), false, ws, static_cast<cudaStream_t>(stream),
                    n_candidates);
}

float moe_router_cert_beta(int32_t hidden) { return hidden > 0 ? moe::router_cert_beta(hidden) : 0.0f; }

moe_status moe_forward_hostio(const moe_config* cfg, int32_t T, const uint16_t* h_host,
                              const uint16_t* w_gate, const float* router_bias, const uint16_t* w13,
                              const uint16_t* w2, const uint16_t* w13_shared, const uint16_t* w2_shared,
                              uint16_t* out_host, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_cfg(cfg));
  MOE_TRY(check_T(cfg, T));
  if (T == 0) return MOE_OK;
  if (!h_host || !out_host) return MOE_ERR_INVALID_ARG;
  MOE_TRY(need(w_gate));
  MOE_TRY(opt(router_bias));
  MOE_TRY(need(w13));
  MOE_TRY(need(w2));
  MOE_TRY(check_shared(cfg, w13_shared, w2_shared));
  MOE_TRY(check_ws(cfg, T, ws, ws_bytes));
  if (!moe::gemm_smem_ok()) return MOE_ERR_UNSUPPORTED;
  const Layout L = layout_of(cfg, T);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint16_t* h = at<uint16_t>(ws, L.h_stage);
  uint16_t* out = at<uint16_t>(ws, L.out_stage);
  const size_t bytes = sizeof(uint16_t) * (size_t)T * cfg->hidden;
  if (cudaMemcpyAsync(h, h_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return MOE_ERR_CUDA;
  MOE_TRY(forward_impl(cfg, T, h, w_gate, router_bias, w13, w2, w13_shared, w2_shared, out, ws, s));
  if (cudaMemcpyAsync(out_host, out, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_get_device_status(const void* ws, int32_t* status_out, void* stream) {
  if (!ws || !aligned16(ws) || !status_out) return MOE_ERR_INVALID_ARG;
  int32_t v = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  *status_out = v;
  return (v & MOE_DEV_ERR_MASK) ? MOE_ERR_DEVICE : MOE_OK;
}

moe_status moe_clear_device_status(void* ws, void* stream) {
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  return cudaMemsetAsync(ws, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

}  // extern "C"
