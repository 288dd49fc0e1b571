// Capacity-limited dispatch and stable alignment into padded expert blocks.
//
// Capacity is granted in batch order ("Mixture-of-experts routing and LLM
// repeatability", the Switch capacity rule and in-order filling): expert e
// keeps its first C routes by ascending route id; the others skip it.  Stable
// construction ("Route-Block Membership Selects Packed-AWQ Arithmetic",
// section "Stable construction selected a third trajectory"): segments in
// ascending expert id, routes inside a segment in ascending route id, each
// segment padded with the sentinel R = T*k to a multiple of B.
//
// The rank of a route among the earlier routes of its expert is computed
// without atomics: warp peers by __match_any_sync, per-warp counts scanned
// across the warps of a 1024-route tile, per-tile counts scanned across tiles
// in a single CTA.  All results are integers and unique, so every run and
// every launch shape gives the same bits.
#include <cstdint>


#include "kernels.h"
#include "pdl.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kMaxN = 256;

// unrouted_ok: an entry of -1 marks a route that has no expert (dropped by
// reroute, or not chosen by expert choice); it is skipped without a status bit.
__global__ void __launch_bounds__(1024) dispatch_count_kernel(const int32_t* __restrict__ topk_idx,
                                                              int R, int N, int unrouted_ok,
                                                              int32_t* __restrict__ rank_in_tile,
                                                              int32_t* __restrict__ tile_count,
                                                              int* status) {
  pdl_wait();      // earlier kernels' outputs are visible from here on
  pdl_trigger();
  __shared__ int32_t wc[32][kMaxN + 1];
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 32 * (kMaxN + 1); i += blockDim.x) (&wc[0][0])[i] = 0;
  __syncthreads();
  const int r = blockIdx.x * kDispatchTile + tid;
  const int e = (r < R) ? topk_idx[r] : -1;
  const bool valid = (r < R) && e >= 0 && e < N;
  if (r < R && !valid && !(unrouted_ok && e == -1)) atomicOr(status, kDevErrExpertRange);
  const int key = valid ? e : -1;
  const unsigned peers = __match_any_sync(0xffffffffu, key);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (valid && rank == 0) wc[w][e] = __popc(peers);
  __syncthreads();
  for (int ee = tid; ee < N; ee += blockDim.x) {
    int run = 0;
    for (int ww = 0; ww < 32; ++ww) {
      const int c = wc[ww][ee];
      wc[ww][ee] = run;
      run += c;
    }
    tile_count[(size_t)blockIdx.x * N + ee] = run;
  }
  __syncthreads();
  if (r < R) rank_in_tile[r] = valid ? wc[w][e] + rank : -1;
}

// Block-wide exclusive scan of one int per thread (256 threads).
__device__ int block_exclusive_scan(int v, int* buf, int* total) {
  const int tid = threadIdx.x;
  buf[tid] = v;
  __syncthreads();
  for (int off = 1; off < 256; off <<= 1) {
    const int x = (tid >= off) ? buf[tid - off] : 0;
    __syncthreads();
    buf[tid] += x;
    __syncthreads();
  }
  const int incl = buf[tid];
  *total = buf[255];
  __syncthreads();
  return incl - v;
}

// Capacity left to expert e in this batch: all of it, or for one shard of a
// larger batch what the earlier shards (in token order) did not take
// (expert_offset[e] routes); -1: no limit.
__device__ __forceinline__ int capacity_left(int capacity, const int32_t* __restrict__ expert_offset, int e) {
  if (capacity < 0) return -1;
  return expert_offset ? max(0, capacity - expert_offset[e]) : capacity;
}

// Exclusive scan of v over experts 0..N-1 by warp 0 (N <= 256, 8 per lane);
// out[e] = sum of v[0..e-1], returns the total (to lane 0..31).
__device__ int warp_scan_experts(const int* v, int* out, int N, int lane) {
  int loc[8], sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane * 8 + i;
    loc[i] = e < N ? v[e] : 0;
    sum += loc[i];
  }
  int incl = sum;
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  int run = incl - sum;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane * 8 + i;
    if (e < N) out[e] = run;
    run += loc[i];
  }
  return __shfl_sync(0xffffffffu, incl, 31);
}

// One CTA of kScanThreads threads.  Turns per-tile counts into per-tile
// bases (in place), applies the capacity, lays out the segments.  Thread
// (part p, expert e) owns a contiguous run of route tiles of expert e: it
// sums their counts, and once the parts before it are summed writes each
// tile's base (earlier tiles' counts first, tiles in order); warp 0 then
// scans the experts' padded sizes and drops in expert order.
constexpr int kScanThreads = 1024;
constexpr int kScanParts = 16;

__global__ void __launch_bounds__(kScanThreads) dispatch_scan_kernel(
    int32_t* __restrict__ tile_count, int ntiles, int N, int B, int capacity,
    const int32_t* __restrict__ expert_offset, int R,
    int32_t* __restrict__ seg_off, int32_t* __restrict__ expert_counts, int32_t* __restrict__ num_padded,
    int32_t* __restrict__ num_dropped, int32_t* __restrict__ block_expert,
    int32_t* __restrict__ sorted_route_ids) {
  pdl_wait();      // earlier kernels' outputs are visible from here on
  pdl_trigger();
  __shared__ int part_sum[kScanParts][kMaxN];
  __shared__ int s_pad[kMaxN], s_drop[kMaxN], s_seg[kMaxN], s_tmp[kMaxN];
  __shared__ int blk_off[kMaxN + 1];
  __shared__ int s_rows;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = min(min(kScanThreads / N, kScanParts), max(ntiles, 1));
  const int per = (ntiles + P - 1) / P;
  const int e = tid % N, p = tid / N;
  const bool active = p < P;
  const int t0 = p * per, t1 = min(ntiles, t0 + per);
  constexpr int kBatch = 8;
  if (active) {
    int sum = 0;
    for (int b0 = t0; b0 < t1; b0 += kBatch) {
      int c[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) c[j] = (b0 + j < t1) ? tile_count[(size_t)(b0 + j) * N + e] : 0;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) sum += c[j];
    }
    part_sum[p][e] = sum;
  }
  __syncthreads();
  if (active) {
    int run = 0;
    for (int q = 0; q < p; ++q) run += part_sum[q][e];
    for (int b0 = t0; b0 < t1; b0 += kBatch) {
      int c[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) c[j] = (b0 + j < t1) ? tile_count[(size_t)(b0 + j) * N + e] : 0;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (b0 + j < t1) {
          tile_count[(size_t)(b0 + j) * N + e] = run;
          run += c[j];
        }
      }
    }
  }
  if (tid < N) {
    int load = 0;
    for (int q = 0; q < P; ++q) load += part_sum[q][tid];
    const int cap_e = capacity_left(capacity, expert_offset, tid);
    const int kept = cap_e < 0 ? load : min(load, cap_e);
    s_pad[tid] = (kept + B - 1) / B * B;
    s_drop[tid] = load - kept;
    expert_counts[tid] = kept;
    s_tmp[tid] = kept;
  }
  __syncthreads();
  if (warp == 0) {
    const int rows = warp_scan_experts(s_pad, s_seg, N, lane);
    const int drops = warp_scan_experts(s_drop, s_drop, N, lane);
    if (lane == 0) {
      s_rows = rows;
      *num_padded = rows;
      if (num_dropped) *num_dropped = drops;
    }
  }
  __syncthreads();
  const int total_rows = s_rows;
  if (tid < N) {
    const int seg = s_seg[tid];
    seg_off[tid] = seg;
    for (int j = s_tmp[tid]; j < s_pad[tid]; ++j) sorted_route_ids[seg + j] = R;
    blk_off[tid] = seg / B;
  }
  if (tid == 0) blk_off[N] = total_rows / B;
  __syncthreads();
  // block b belongs to the last expert whose first block is <= b
  const int nb = total_rows / B;
  for (int b = tid; b < nb; b += blockDim.x) {
    // largest e in [0, N) with blk_off[e] <= b; it has blk_off[e+1] > b, so
    // empty segments (equal offsets) are skipped
    int lo = 0, hi = N;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (blk_off[mid] <= b) lo = mid; else hi = mid;
    }
    block_expert[b] = lo;
  }
}

__global__ void __launch_bounds__(1024) dispatch_scatter_kernel(
    const int32_t* __restrict__ topk_idx, int R, int N, int capacity, const int32_t* __restrict__ expert_offset,
    const int32_t* __restrict__ rank_in_tile, const int32_t* __restrict__ tile_base,
    const int32_t* __restrict__ seg_off, uint8_t* __restrict__ route_kept,
    int32_t* __restrict__ route_pos, int32_t* __restrict__ sorted_route_ids) {
  pdl_wait();      // earlier kernels' outputs are visible from here on
  pdl_trigger();
  const int r = blockIdx.x * kDispatchTile + threadIdx.x;
  if (r >= R) return;
  const int e = topk_idx[r];
  if (e < 0 || e >= N) {
    route_kept[r] = 0;
    route_pos[r] = -1;
    return;
  }
  const int rank = tile_base[(size_t)blockIdx.x * N + e] + rank_in_tile[r];
  const int cap_e = capacity_left(capacity, expert_offset, e);
  const bool kept = cap_e < 0 || rank < cap_e;
  route_kept[r] = kept ? 1 : 0;
  if (kept) {
    const int pos = seg_off[e] + rank;
    route_pos[r] = pos;
    sorted_route_ids[pos] = r;
  } else {
    route_pos[r] = -1;
  }
}

// Grouped-GEMM tile list from the padded blocks, by one CTA: each expert
// segment is cut into tiles of tile_rows rows from its start.  Rejects (no
// tiles, status bit) a block list that is not sorted by expert or out of
// range.
__device__ __forceinline__ void build_tiles_block(const int32_t* __restrict__ block_expert,
                                                  const int32_t* __restrict__ num_padded,
                                                  const int32_t* __restrict__ sorted_route_ids, int R, int N,
                                                  int B, long long max_rows, const TileListOut& L,
                                                  int* status) {
  __shared__ int buf[256];
  __shared__ int s_first[kMaxN], s_last[kMaxN];
  __shared__ int s_bad;
  const int P = *num_padded;
  const bool bad_count = P < 0 || (long long)P > max_rows || (P % B) != 0;
  const int nb = bad_count ? 0 : P / B;
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    s_first[e] = 0;
    s_last[e] = 0;
  }
  if (threadIdx.x == 0) s_bad = bad_count ? 1 : 0;
  __syncthreads();
  // one pass over the blocks checks the order and marks where each expert's
  // blocks begin and end (an expert with no block keeps an empty range)
  // (four blocks per thread and round: their loads are issued together)
  constexpr int kPassUnroll = 4;
  for (int b0 = threadIdx.x; b0 < nb; b0 += kPassUnroll * blockDim.x) {
    int e[kPassUnroll], prev[kPassUnroll], next[kPassUnroll];
#pragma unroll
    for (int j = 0; j < kPassUnroll; ++j) {
      const int b = b0 + j * blockDim.x;
      e[j] = b < nb ? block_expert[b] : 0;
      prev[j] = (b < nb && b > 0) ? block_expert[b - 1] : -1;
      next[j] = b + 1 < nb ? block_expert[b + 1] : N;
    }
#pragma unroll
    for (int j = 0; j < kPassUnroll; ++j) {
      const int b = b0 + j * blockDim.x;
      if (b >= nb) continue;
      if (e[j] < 0 || e[j] >= N || prev[j] > e[j]) {
        s_bad = 1;
        continue;
      }
      if (prev[j] != e[j]) s_first[e[j]] = b;
      if (next[j] != e[j]) s_last[e[j]] = b + 1;
    }
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) {
      *L.num_tiles = 0;
      if (L.next_item) *L.next_item = 0;
      atomicOr(status, kDevErrBadBlocks);
    }
    return;
  }
  const int e = threadIdx.x;
  const int first = e < N ? s_first[e] : 0, last = e < N ? s_last[e] : 0;
  const int rows = (last - first) * B;
  // rows up to the segment's last route (the padding sentinels trail it),
  // eight rows from the end per round trip
  int used = rows;
  while (used > 0) {
    const int n = min(8, used);
    int r[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) r[j] = j < n ? sorted_route_ids[first * B + used - 1 - j] : -1;
    int found = -1;
#pragma unroll
    for (int j = 7; j >= 0; --j)
      if (j < n && r[j] >= 0 && r[j] < R) found = j;
    if (found >= 0) {
      used -= found;
      break;
    }
    used -= n;
  }
  const int tile_rows = L.tile_rows;
  const int nt = segment_tiles(rows, tile_rows);
  int total = 0;
  const int off = block_exclusive_scan(nt, buf, &total);
  for (int j = 0; j < nt; ++j) {
    const int idx = off + j;
    if (idx < L.max_tiles) L.tiles[idx] = segment_tile(e, first * B, rows, used, tile_rows, nt, j, off);
  }
  if (threadIdx.x == 0) {
    *L.num_tiles = min(total, L.max_tiles);
    if (L.next_item) *L.next_item = 0;
  }
}

// x_perm[p] = h[r / k] for padded row p holding route r, zeros for the
// sentinel: the routed token rows in expert-segment order, so that the W13
// GEMM loads whole 128-row tiles.  One warp per row (warps w0, w0 + warps,
// ...), 16-byte accesses, up to eight pieces per lane loaded before they are
// stored, the next row's route id in flight meanwhile.
__device__ __forceinline__ void gather_rows_warps(const uint16_t* __restrict__ h,
                                                  const int32_t* __restrict__ sorted_route_ids,
                                                  long long P, int k, int R, int H,
                                                  uint16_t* __restrict__ x_perm, long long w0,
                                                  long long warps) {
  const int lane = threadIdx.x & 31;
  const int chunks = H / 8;
  int r = w0 < P ? sorted_route_ids[w0] : -1;
  for (long long row = w0; row < P; row += warps) {
    const long long nrow = row + warps;
    const int rn = nrow < P ? sorted_route_ids[nrow] : -1;
    uint4* dst = reinterpret_cast<uint4*>(x_perm + row * H);
    if (r >= 0 && r < R) {
      const uint4* src = reinterpret_cast<const uint4*>(h + (size_t)(r / k) * H);
      for (int c0 = lane; c0 < chunks; c0 += 8 * 32) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (c0 + 32 * u < chunks) v[u] = __ldg(src + c0 + 32 * u);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (c0 + 32 * u < chunks) dst[c0 + 32 * u] = v[u];
      }
    } else {
      for (int c = lane; c < chunks; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
    }
    r = rn;
  }
}

// The same x_perm token by token (warps w0, w0 + warps, ... over the T tokens,
// then the padded rows): warp per token, h[t] read once from DRAM
// and copied (from L1) to the padded row route_pos[t k + j] of each kept
// slot; then zeros in the padding rows.  When h is larger than L2 the
// segment-order gather fetches a token's row once per slot.
__device__ __forceinline__ void scatter_rows_warps(const uint16_t* __restrict__ h,
                                                   const int32_t* __restrict__ route_pos,
                                                   const int32_t* __restrict__ sorted_route_ids,
                                                   long long P, int k, int T, int H,
                                                   uint16_t* __restrict__ x_perm, long long w0,
                                                   long long warps) {
  const long long R = (long long)T * k;
  const int lane = threadIdx.x & 31;
  const int chunks = H / 8;
  for (long long item = w0; item < T + P; item += warps) {
    if (item < T) {
      // each 16-byte piece of the row is loaded once and stored to every
      // kept slot; lane l holds the padded row of slot g * 32 + l, for the
      // slot groups g of 32 (one group for token choice, k <= 16)
      const uint4* src = reinterpret_cast<const uint4*>(h + (size_t)item * H);
      auto slot_row = [&](int j) -> long long {
        const long long p = j < k ? route_pos[item * k + j] : -1;
        return (p < 0 || p >= P) ? -1 : p;   // dropped
      };
      const long long p0 = slot_row(lane);
      const unsigned kept0 = __ballot_sync(0xffffffffu, p0 >= 0);
      // (the loop bounds are the same in every lane: the shuffles below need the whole warp)
      for (int base = 0; base < chunks; base += 4 * 32) {
        const int c0 = base + lane;
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (c0 + u * 32 < chunks) v[u] = __ldg(src + c0 + u * 32);
        for (int g = 0; g * 32 < k; ++g) {
          const long long my_p = g == 0 ? p0 : slot_row(g * 32 + lane);
          const unsigned kept = g == 0 ? kept0 : __ballot_sync(0xffffffffu, my_p >= 0);
          for (unsigned m = kept; m; m &= m - 1) {
            const long long p = __shfl_sync(0xffffffffu, my_p, __ffs(m) - 1);
            uint4* dst = reinterpret_cast<uint4*>(x_perm + p * H);
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (c0 + u * 32 < chunks) dst[c0 + u * 32] = v[u];
          }
        }
      }
    } else {
      const long long row = item - T;
      const int r = sorted_route_ids[row];
      if (r < 0 || r >= R) {
        uint4* dst = reinterpret_cast<uint4*>(x_perm + row * H);
        for (int c = lane; c < chunks; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
      }
    }
  }
}

// The GEMM tile lists and the routed token rows in one launch: CTAs below
// `lists` each build one tile list (CTA 0 list a, CTA 1 list b); the others
// copy the rows (kRows 1: in padded-row order, 2: token by token, 0: none).
// The grid is sized to be resident at once, so the GEMM may launch early:
// its CTAs set up on the SMs this grid releases and wait for it to finish.
template <int kRows>
__global__ void __launch_bounds__(256) tiles_rows_kernel(const int32_t* __restrict__ block_expert,
                                                         const int32_t* __restrict__ num_padded,
                                                         const int32_t* __restrict__ sorted_route_ids,
                                                         int k, int T, int N, int B, long long max_rows,
                                                         int lists, TileListOut a, TileListOut b,
                                                         int* status, const uint16_t* __restrict__ h,
                                                         const int32_t* __restrict__ route_pos, int H,
                                                         uint16_t* __restrict__ x_perm) {
  pdl_wait();      // earlier kernels' outputs are visible from here on
  pdl_trigger();
  const int R = T * k;
  if ((int)blockIdx.x < lists) {
    build_tiles_block(block_expert, num_padded, sorted_route_ids, R, N, B, max_rows, blockIdx.x == 0 ? a : b,
                      status);
    return;
  }
  if (kRows == 0) return;
  const long long P = min((long long)*num_padded, max_rows);
  const long long w0 = (long long)(blockIdx.x - lists) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const long long warps = (long long)(gridDim.x - lists) * (blockDim.x >> 5);
  if (kRows == 1)
    gather_rows_warps(h, sorted_route_ids, P, k, R, H, x_perm, w0, warps);
  else
    scatter_rows_warps(h, route_pos, sorted_route_ids, P, k, T, H, x_perm, w0, warps);
}

// Dispatch, alignment and both GEMM tile lists of a batch of at most 1024
// routes in one CTA (decode): the same integers as dispatch_count, _scan,
// _scatter and build_tiles (ranks by warp match, per-warp counts added in
// warp order, segment and tile offsets by ordered scans), in one launch.
constexpr int kSmallDispatchMaxR = 1024;


// The body: one CTA of at least R threads (full warps), thread r handles
// route r.  topk_idx is read with plain loads (the decode front writes it in
// the same kernel).
__device__ __forceinline__ void dispatch_small_block(
    const int32_t* topk_idx, int R, int N, int B, int capacity, uint8_t* __restrict__ route_kept,
    int32_t* route_pos, int32_t* __restrict__ sorted_route_ids, int32_t* __restrict__ block_expert,
    int32_t* __restrict__ num_padded, int32_t* __restrict__ expert_counts, int32_t* __restrict__ num_dropped,
    const TileListOut& la, const TileListOut& lb, int* status, int32_t* pos_smem = nullptr) {
  __shared__ int wc[32][kMaxN + 1];
  __shared__ int kept_s[kMaxN], pad_s[kMaxN], drop_s[kMaxN], nta[kMaxN], ntb[kMaxN];
  __shared__ int seg[kMaxN], offa[kMaxN], offb[kMaxN];
  __shared__ int s_rows, s_drop, s_ta, s_tb;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  // warps holding routes (R <= 1024 = 32 warps): only their counts are used
  const int rw = (R + 31) >> 5;
  for (int i = tid; i < rw * (kMaxN + 1); i += blockDim.x) (&wc[0][0])[i] = 0;
  __syncthreads();
  const int r = tid;
  const int e = (r < R) ? topk_idx[r] : -1;
  const bool valid = (r < R) && e >= 0 && e < N;
  if (r < R && !valid) atomicOr(status, kDevErrExpertRange);
  const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (valid && rank == 0) wc[w][e] = __popc(peers);
  __syncthreads();
  for (int x = tid; x < N; x += blockDim.x) {
    int run = 0;
    for (int ww = 0; ww < rw; ++ww) {
      const int c = wc[ww][x];
      wc[ww][x] = run;
      run += c;
    }
    const int kept = capacity < 0 ? run : min(run, capacity);
    const int padded = (kept + B - 1) / B * B;
    kept_s[x] = kept;
    pad_s[x] = padded;
    drop_s[x] = run - kept;
    nta[x] = segment_tiles(padded, la.tile_rows);
    ntb[x] = segment_tiles(padded, lb.tile_rows);
    expert_counts[x] = kept;
  }
  __syncthreads();
  if (w == 0) {
    const int rows = warp_scan_experts(pad_s, seg, N, lane);
    const int ta = warp_scan_experts(nta, offa, N, lane);
    const int tb = warp_scan_experts(ntb, offb, N, lane);
    int dsum = 0;
    for (int x = lane; x < N; x += 32) dsum += drop_s[x];
    for (int off = 16; off > 0; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
    if (lane == 0) {
      s_rows = rows;
      s_drop = dsum;
      s_ta = ta;
      s_tb = tb;
    }
  }
  __syncthreads();
  if (r < R) {
    int p = -1;
    if (valid) {
      const int rk = wc[w][e] + rank;
      const bool kept = capacity < 0 || rk < capacity;
      route_kept[r] = kept ? 1 : 0;
      if (kept) {
        p = seg[e] + rk;
        sorted_route_ids[p] = r;
      }
    } else {
      route_kept[r] = 0;
    }
    route_pos[r] = p;
    if (pos_smem) pos_smem[r] = p;   // the caller's copy of the rows reads it here
  }
  for (int x = tid; x < N; x += blockDim.x) {
    for (int j = kept_s[x]; j < pad_s[x]; ++j) sorted_route_ids[seg[x] + j] = R;
    for (int b = seg[x] / B; b < (seg[x] + pad_s[x]) / B; ++b) block_expert[b] = x;
    for (int j = 0; j < nta[x]; ++j) {
      const int idx = offa[x] + j;
      if (idx < la.max_tiles)
        la.tiles[idx] = segment_tile(x, seg[x], pad_s[x], kept_s[x], la.tile_rows, nta[x], j, offa[x]);
    }
    for (int j = 0; j < ntb[x]; ++j) {
      const int idx = offb[x] + j;
      if (idx < lb.max_tiles)
        lb.tiles[idx] = segment_tile(x, seg[x], pad_s[x], kept_s[x], lb.tile_rows, ntb[x], j, offb[x]);
    }
  }
  if (tid == 0) {
    *num_padded = s_rows;
    *num_dropped = s_drop;
    *la.num_tiles = min(s_ta, la.max_tiles);
    *lb.num_tiles = min(s_tb, lb.max_tiles);
    if (la.next_item) *la.next_item = 0;
    if (lb.next_item) *lb.next_item = 0;
  }
}

__global__ void __launch_bounds__(kSmallDispatchMaxR) dispatch_small_kernel(
    const int32_t* __restrict__ topk_idx, int R, int N, int B, int capacity,
    uint8_t* __restrict__ route_kept, int32_t* __restrict__ route_pos,
    int32_t* __restrict__ sorted_route_ids, int32_t* __restrict__ block_expert,
    int32_t* __restrict__ num_padded, int32_t* __restrict__ expert_counts,
    int32_t* __restrict__ num_dropped, const TileListOut la, const TileListOut lb, int* status) {
  pdl_wait();      // earlier kernels' outputs are visible from here on
  pdl_trigger();
  dispatch_small_block(topk_idx, R, N, B, capacity, route_kept, route_pos, sorted_route_ids, block_expert,
                       num_padded, expert_counts, num_dropped, la, lb, status);
}

// ------------------------------------------------------------------------
// Decode finish: for a few tokens, everything between the router's chunk sums
// and the W13 GEMM in one CTA: the logits (chunk sums added in ascending
// chunk order, then the bias, exactly as router_reduce_kernel), the same
// top-k and gates, the same dispatch body with both tile lists, and the
// routed token rows of x_perm.
constexpr int kFinishThreads = 512;
constexpr int kFinishMaxT = 2;
constexpr int kRowPieces = 4;   // token-row pieces per thread requested at the start

__global__ void __launch_bounds__(kFinishThreads, 1) decode_finish_kernel(
    const float* __restrict__ part, const uint16_t* __restrict__ h, const float* __restrict__ bias, int T, int H,
    int N, int k, int B, int capacity, int32_t* topk_idx, float* __restrict__ gates,
    uint8_t* __restrict__ route_kept, int32_t* route_pos, int32_t* __restrict__ sorted_route_ids,
    int32_t* __restrict__ block_expert, int32_t* __restrict__ num_padded, int32_t* __restrict__ expert_counts,
    int32_t* __restrict__ num_dropped, const TileListOut la, const TileListOut lb,
    uint16_t* __restrict__ x_perm, long long max_rows, int* status) {
  pdl_wait();      // earlier kernels' outputs are visible from here on
  // one CTA: the GEMM's CTAs may set up on the other SMs meanwhile (they
  // wait for this kernel to finish)
  pdl_trigger();
  __shared__ float lrow[kFinishMaxT][kMaxN];
  // the routes' experts and padded rows stay in shared memory for the steps
  // of this CTA that read them (their global copies are for later kernels)
  __shared__ int32_t s_idx[kFinishMaxT * 16];
  __shared__ float s_gate[kFinishMaxT * 16];
  __shared__ int32_t s_pos[kFinishMaxT * 16];
  const int C = (H + kRouterChunk - 1) / kRouterChunk;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the token rows do not depend on the routing: with at most four 16-byte
  // pieces per thread they are requested now, and stored to their routes'
  // padded rows once the dispatch has placed them
  const int pieces = H / 8;
  const bool early_rows = T * pieces <= kRowPieces * kFinishThreads;
  uint4 rowv[kRowPieces];
#pragma unroll
  for (int u = 0; u < kRowPieces; ++u) {
    const int x = tid + u * kFinishThreads;
    if (early_rows && x < T * pieces)
      rowv[u] = __ldg(reinterpret_cast<const uint4*>(h + (size_t)(x / pieces) * H) + x % pieces);
  }
  for (int x = tid; x < T * N; x += blockDim.x) {
    // the chunk sums (and the bias) requested sixteen at a time, then added
    // in ascending chunk order
    const int t = x / N, e = x % N;
    const float* pe = part + (size_t)t * C * N + e;
    const float be = bias ? bias[e] : 0.0f;
    float total = 0.0f;
    for (int c0 = 0; c0 < C; c0 += 16) {
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = c0 + j < C ? pe[(size_t)(c0 + j) * N] : 0.0f;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (c0 + j < C) total = total + v[j];
    }
    if (bias) total = total + be;
    lrow[t][e] = total;
  }
  __syncthreads();
  if (warp < T) sel::topk_select_warp(lrow[warp], N, k, lane, s_idx + warp * k, s_gate + warp * k);
  __syncthreads();
  const int R = T * k;
  if (tid < R) {
    topk_idx[tid] = s_idx[tid];
    gates[tid] = s_gate[tid];
  }
  dispatch_small_block(s_idx, R, N, B, capacity, route_kept, route_pos, sorted_route_ids, block_expert,
                       num_padded, expert_counts, num_dropped, la, lb, status, s_pos);
  __syncthreads();
  if (early_rows) {
    // each requested piece to the padded row of each kept route of its token
#pragma unroll
    for (int u = 0; u < kRowPieces; ++u) {
      const int x = tid + u * kFinishThreads;
      if (x < T * pieces) {
        const int t = x / pieces, q = x % pieces;
        for (int j = 0; j < k; ++j) {
          const long long p = s_pos[t * k + j];
          if (p >= 0 && p < max_rows) *(reinterpret_cast<uint4*>(x_perm + p * H) + q) = rowv[u];
        }
      }
    }
    return;
  }
  // the routed token rows (padding rows feed only MMA columns that are never
  // stored), four 16-byte pieces per thread and round, loads before stores
  const int total = R * pieces;
  for (int x0 = tid; x0 < total; x0 += 4 * blockDim.x) {
    uint4 v[4];
    long long dst[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int x = x0 + u * blockDim.x;
      dst[u] = -1;
      if (x < total) {
        const int r = x / pieces, q = x % pieces;
        const long long p = s_pos[r];
        if (p >= 0 && p < max_rows) {
          v[u] = __ldg(reinterpret_cast<const uint4*>(h + (size_t)(r / k) * H) + q);
          dst[u] = p * H + (long long)q * 8;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (dst[u] >= 0) *reinterpret_cast<uint4*>(x_perm + dst[u]) = v[u];
  }
}

}  // namespace

void launch_dispatch(const int32_t* topk_idx, int T, int N, int k, int B, int capacity,
                     uint8_t* route_kept, int32_t* route_pos, int32_t* sorted_route_ids,
                     int32_t* block_expert, int32_t* num_padded, int32_t* expert_counts,
                     int32_t* num_dropped, int32_t* rank_in_tile, int32_t* tile_count,
                     int32_t* seg_off, int* status, cudaStream_t s, const int32_t* expert_offset) {
  const int R = T * k;
  const int ntiles = (R + kDispatchTile - 1) / kDispatchTile;
  launch_pdl(dispatch_count_kernel, dim3(ntiles), dim3(kDispatchTile), 0, s, topk_idx, R, N, 0, rank_in_tile, tile_count,
                                                         status);
  launch_pdl(dispatch_scan_kernel, dim3(1), dim3(kScanThreads), 0, s, tile_count, ntiles, N, B, capacity, expert_offset, R,
             seg_off, expert_counts, num_padded, num_dropped, block_expert, sorted_route_ids);
  launch_pdl(dispatch_scatter_kernel, dim3(ntiles), dim3(kDispatchTile), 0, s, topk_idx, R, N, capacity,
             expert_offset, rank_in_tile, tile_count, seg_off, route_kept, route_pos, sorted_route_ids);
}

void launch_dispatch_routes(const int32_t* route_expert, int R, int N, int B, uint8_t* route_kept,
                            int32_t* route_pos, int32_t* sorted_route_ids, int32_t* block_expert,
                            int32_t* num_padded, int32_t* expert_counts, int32_t* rank_in_tile,
                            int32_t* tile_count, int32_t* seg_off, int* status, cudaStream_t s) {
  const int ntiles = (R + kDispatchTile - 1) / kDispatchTile;
  launch_pdl(dispatch_count_kernel, dim3(ntiles), dim3(kDispatchTile), 0, s, route_expert, R, N, 1, rank_in_tile, tile_count,
                                                         status);
  launch_pdl(dispatch_scan_kernel, dim3(1), dim3(kScanThreads), 0, s, tile_count, ntiles, N, B, -1, (const int32_t*)nullptr, R,
             seg_off, expert_counts, num_padded, (int32_t*)nullptr, block_expert, sorted_route_ids);
  launch_pdl(dispatch_scatter_kernel, dim3(ntiles), dim3(kDispatchTile), 0, s, route_expert, R, N, -1,
             (const int32_t*)nullptr, rank_in_tile, tile_count, seg_off, route_kept, route_pos, sorted_route_ids);
}

void launch_dispatch_reroute(const int32_t* topk_idx, const float* logits, int T, int N, int k, int B,
                             int capacity, uint8_t* route_kept, int32_t* route_expert,
                             int32_t* route_pos, int32_t* sorted_route_ids, int32_t* block_expert,
                             int32_t* num_padded, int32_t* expert_counts, int32_t* num_dropped,
                             int32_t* num_rerouted, int32_t* rank_in_tile, int32_t* tile_count,
                             int32_t* seg_off, const RerouteScratch& sc, int* status, const PathOpts& o,
                             cudaStream_t s) {
  const int R = T * k;
  const int ntiles = (R + kDispatchTile - 1) / kDispatchTile;
  // phase one: ranks and the per-expert kept counts of the drop rule
  launch_pdl(dispatch_count_kernel, dim3(ntiles), dim3(kDispatchTile), 0, s, topk_idx, R, N, 0, rank_in_tile, tile_count,
                                                         status);
  launch_pdl(dispatch_scan_kernel, dim3(1), dim3(kScanThreads), 0, s, tile_count, ntiles, N, B, capacity, (const int32_t*)nullptr, R,
             seg_off, expert_counts, num_padded, (int32_t*)nullptr, block_expert, sorted_route_ids);
  // phase two, then the stable layout of the final assignment
  launch_reroute(topk_idx, logits, T, N, k, capacity, rank_in_tile, tile_count, expert_counts, sc,
                 route_expert, num_dropped, num_rerouted, status, o, s);
  launch_dispatch_routes(route_expert, R, N, B, route_kept, route_pos, sorted_route_ids, block_expert,
                         num_padded, expert_counts, rank_in_tile, tile_count, seg_off, status, s);
}

bool dispatch_small_ok(long long R) { return R <= kSmallDispatchMaxR; }

void launch_dispatch_small(const int32_t* topk_idx, int R, int N, int B, int capacity, uint8_t* route_kept,
                           int32_t* route_pos, int32_t* sorted_route_ids, int32_t* block_expert,
                           int32_t* num_padded, int32_t* expert_counts, int32_t* num_dropped,
                           const TileListOut& la, const TileListOut& lb, int* status, cudaStream_t s) {
  launch_pdl(dispatch_small_kernel, dim3(1), dim3(kSmallDispatchMaxR), 0, s, topk_idx, R, N, B, capacity,
             route_kept, route_pos, sorted_route_ids, block_expert, num_padded, expert_counts, num_dropped, la, lb,
             status);
}

// The caller's path flags may turn the two-launch front off (the bits are
// the same either way).
bool decode_front_ok(int T, int H, int N, int k, uint32_t path_flags) {
  if (path_flags & kPathNoDecodeFront) return false;
  return T >= 1 && T <= kFinishMaxT && H % 8 == 0 && N <= kMaxN && k <= 16 && T * k <= kFinishThreads;
}

void launch_decode_front(const uint16_t* h, const uint16_t* w_gate, const float* bias, float* part, int T, int H,
                         int N, int k, int B, int capacity, int32_t* topk_idx, float* gates, uint8_t* route_kept,
                         int32_t* route_pos, int32_t* sorted_route_ids, int32_t* block_expert, int32_t* num_padded,
                         int32_t* expert_counts, int32_t* num_dropped, const TileListOut& la,
                         const TileListOut& lb, uint16_t* x_perm, int64_t max_rows, int* status, cudaStream_t s) {
  launch_router_partials(h, w_gate, part, T, H, N, s);
  launch_pdl(decode_finish_kernel, dim3(1), dim3(kFinishThreads), 0, s, (const float*)part, h, bias, T, H, N, k, B,
             capacity, topk_idx, gates, route_kept, route_pos, sorted_route_ids, block_expert, num_padded,
             expert_counts, num_dropped, la, lb, x_perm, (long long)max_rows, status);
}

void launch_tiles_and_rows(const int32_t* block_expert, const int32_t* num_padded,
                           const int32_t* sorted_route_ids, int k, int T, int N, int B, int64_t max_rows,
                           const TileListOut* a, const TileListOut* b, int* status, int row_mode,
                           const uint16_t* h, const int32_t* route_pos, int H, uint16_t* x_perm,
                           cudaStream_t s) {
  const int lists = a ? (b ? 2 : 1) : 0;
  auto kernel = row_mode == 1 ? tiles_rows_kernel<1> : (row_mode == 2 ? tiles_rows_kernel<2> : tiles_rows_kernel<0>);
  int row_blocks = 0;
  if (row_mode != 0) {
    // every CTA resident at once (SMs x resident CTAs per SM, less the list
    // CTAs), each row warp then striding over the rows
    static int cache[64][3] = {};   // per device and row mode: SMs x resident CTAs
    int dev = 0;
    cudaGetDevice(&dev);
    int cap = (dev >= 0 && dev < 64) ? cache[dev][row_mode] : 0;
    if (cap <= 0) {
      int sms = 0, per = 0;
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, 256, 0);
      cap = (sms > 0 ? sms : 1) * (per > 0 ? per : 1);
      if (dev >= 0 && dev < 64) cache[dev][row_mode] = cap;
    }
    cap = cap > lists ? cap - lists : 1;   // the list CTAs take resident slots too
    const long long items = row_mode == 2 ? (long long)T + max_rows : (long long)max_rows;
    const long long want = (items + 7) / 8;
    row_blocks = (int)(want < cap ? (want > 0 ? want : 1) : cap);
  }
  if (lists + row_blocks == 0) return;
  const TileListOut la = a ? *a : TileListOut{};
  const TileListOut lb = b ? *b : la;
  launch_pdl(kernel, dim3(lists + row_blocks), dim3(256), 0, s, block_expert, num_padded, sorted_route_ids, k, T,
             N, B, (long long)max_rows, lists, la, lb, status, h, route_pos, H, x_perm);
}

}  // namespace moe
