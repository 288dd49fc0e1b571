// Grouped SwiGLU expert GEMMs on the 5th-generation tensor cores (tcgen05).
//
// For each padded expert segment produced by the stable alignment
// ("Route-Block Membership Selects Packed-AWQ Arithmetic", "The bookkeeping
// before the matrix multiplication"), token tiles of BN rows run
//   W13: [g | u] = X . W13_e  ->  a = bf16(silu(g) * u)      (X = x_perm rows)
//   W2 : y = a . W2_e         ->  y_perm (fp32 accumulation, stored as bf16)
// The weights are operand A (M = 128 output features, MN-major straight from
// the [K, features] layout), the tokens operand B (N = BN rows, K-major; BN =
// 128 for W13, 256 for W2).  Every tile of every batch runs the same
// instruction sequence: one tile shape per GEMM, K from 0 to the end in steps
// of 64 (four K=16 MMAs each), fp32
// accumulation in TMEM, no split-K and no atomics, so the bits of a token's
// row depend only on that row and the expert's weights ("Why temperature=0
// Still Gives Different Answers: Batch Invariance": one tile configuration,
// no split-K).  Which padded block a route lands in changes nothing, unlike
// the split/non-split schedule classes of the packed kernel that page studies.
//
// Persistent kernel, one CTA per SM, 10 warps:
//   warp 0      TMA producer (weight boxes and the token tile)
//   warp 1      TMEM allocation, one elected thread issues tcgen05.mma
//   warps 2..9  epilogue: tcgen05.ld from TMEM, SiLU*up or fp32 store (two
//               warps per TMEM lane quarter, one half of the columns each)
// Smem stages are guarded by full/empty mbarriers, the TMEM accumulators by
// tmem_full/tmem_empty; where two buffers fit in the 512 TMEM columns (W2)
// the epilogue of one tile overlaps the MMAs of the next.  Every wait is bounded (see mbar_wait).
#include <cuda_bf16.h>
#include <cstdint>

#include "gemm.h"
#include "pdl.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBK = 64;                             // K per stage: one 128-byte swizzle row
constexpr uint32_t kBoxBytes = 64 * 64 * 2;         // 64 K rows x 64 features of bf16
constexpr int kEpiWarps = 8;                        // two per TMEM lane quarter, one column half each
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr int kSmallRows = 32;                      // token box when a tile has <= 32 routed rows
static_assert(kSmallRows == kDecodeMaxT, "the decode instances take small tiles only");
constexpr uint32_t kStageBudget = 192 * 1024;       // shared memory for the operand stages
// Work items reach the MMA issuer and the epilogue warps through a ring of
// this many slots, filled by the producer (which fetches them).
constexpr int kItemRing = 8;

constexpr uint32_t pow2_at_least(uint32_t x) {
  uint32_t p = 32;
  while (p < x) p <<= 1;
  return p;
}

// BN = token rows per tile (the N of every MMA): one fixed value per kernel
// instance, the same for every batch.
template <bool kW13, int BN>
struct GemmCfg {
  static constexpr uint32_t kABytes = kW13 ? 4 * kBoxBytes : 2 * kBoxBytes;
  static constexpr uint32_t kBTileBytes = BN * kBK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBTileBytes;
  static constexpr int kStages = (int)(kStageBudget / kStageBytes) < 6 ? (int)(kStageBudget / kStageBytes) : 6;
  static constexpr uint32_t kAccCols = kW13 ? 2 * BN : BN;            // one accumulator buffer
  static constexpr int kNumAcc = (2 * kAccCols <= 512) ? 2 : 1;       // TMEM double buffering
  static constexpr uint32_t kTmemCols = pow2_at_least(kNumAcc * kAccCols);
  static constexpr uint32_t kBarBytes = 256;
  static constexpr uint32_t kSmemBytes = kStages * kStageBytes + kBarBytes + 1024;
  // M = 128 features, N = BN token rows; A (weights) MN-major, B (tokens) K-major.
  static constexpr uint32_t kIdesc = idesc_bf16(kTileFeat, BN, true, false);
  static constexpr uint32_t kIdescSmall = idesc_bf16(kTileFeat, kSmallRows, true, false);
};

struct TileInfo {
  int expert, row0, rows, valid;
};

template <int BN>
__device__ __forceinline__ TileInfo tile_of(const GemmArgs& a, int ti) {
  TileInfo t;
  if (a.identity_T) {
    t.expert = 0;
    t.row0 = ti * BN;
    t.rows = min(BN, a.identity_T - t.row0);
    t.valid = t.rows;
  } else {
    const GemmTile g = a.tiles[ti];
    t.expert = g.expert;
    t.row0 = g.row0;
    t.rows = g.rows;
    t.valid = g.valid;
  }
  return t;
}

// Work item -> (feature tile, token tile).  Items of one expert are
// contiguous; inside an expert they run in groups of G feature tiles x all of
// the expert's token tiles, G sized so that one wave of CTAs shares its weight
// and token tiles through L2.  Only the order of tiles changes with the batch,
// never the arithmetic of a tile.
struct Work {
  int f;
  TileInfo t;
};

template <int BN>
__device__ __forceinline__ Work work_of(const GemmArgs& a, int item, int num_tiles, int nf) {
  int first = 0, count = num_tiles;
  if (!a.identity_T) {
    const GemmTile g = a.tiles[item / nf];
    first = g.first;
    count = g.count;
  }
  const int l = item - first * nf;
  const int waves = a.concurrent;  // work units that run at the same time
  const int G = max(1, min(nf, (waves + count - 1) / count));
  const int grp = l / (count * G);
  const int gsz = min(G, nf - grp * G);
  const int lin = l - grp * count * G;
  Work w;
  w.f = grp * G + lin % gsz;
  w.t = tile_of<BN>(a, first + lin / gsz);
  return w;
}

// A slot of the item ring: the item and the tile it names (item -1: no
// more items).  The producer that fetches an item fills its slot, so the
// MMA issuer and the epilogue warps read the tile from shared memory.
struct ItemSlot {
  int item, f, expert, row0, valid, pad[3];
};

template <int BN>
__device__ __forceinline__ ItemSlot slot_of(const GemmArgs& a, int item, int total, int num_tiles, int nf) {
  ItemSlot v{};
  v.item = -1;
  if (item >= 0 && item < total) {
    const Work w = work_of<BN>(a, item, num_tiles, nf);
    v.item = item;
    v.f = w.f;
    v.expert = w.t.expert;
    v.row0 = w.t.row0;
    v.valid = w.t.valid;
  }
  return v;
}

__device__ __forceinline__ ItemSlot shfl_slot(const ItemSlot& v) {
  ItemSlot r{};
  r.item = __shfl_sync(0xffffffffu, v.item, 0);
  r.f = __shfl_sync(0xffffffffu, v.f, 0);
  r.expert = __shfl_sync(0xffffffffu, v.expert, 0);
  r.row0 = __shfl_sync(0xffffffffu, v.row0, 0);
  r.valid = __shfl_sync(0xffffffffu, v.valid, 0);
  return r;
}

template <bool kW13, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap w_map,
                       const __grid_constant__ CUtensorMap x_map,
                       const __grid_constant__ CUtensorMap x_map_small, const GemmArgs args) {
  using C = GemmCfg<kW13, BN>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem_base;
  __shared__ volatile int s_abort;
  __shared__ __align__(8) uint64_t s_ibar[2 * kItemRing];   // item ring: full, then empty barriers
  __shared__ ItemSlot s_ring[kItemRing];

  const int nfe = args.n_feat_tiles;
  const int unit0 = (int)blockIdx.x;
  const int units = (int)gridDim.x;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * C::kStages;
  const uint32_t tfull0 = empty0 + 8 * C::kStages;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;
  const uint32_t ifull0 = smem_u32(s_ibar), iempty0 = ifull0 + 8 * kItemRing;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ksteps = args.K / kBK;
  const uint64_t wlim = args.wait_ns ? args.wait_ns : kWaitLimitNs;   // pipeline waits

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < C::kNumAcc; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, kEpiWarps * 32);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(ifull0 + 8 * i, 1);
      mbar_init(iempty0 + 8 * i, 1 + kEpiWarps);   // the MMA issuer and each epilogue warp
    }
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s_tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&w_map);
    prefetch_tmap(&x_map);
    prefetch_tmap(&x_map_small);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem_base;
  // The set-up above reads nothing an earlier kernel writes: it overlaps the
  // end of that kernel.  Every CTA of this persistent grid is resident, so
  // the next kernel may launch now (its CTAs wait for this grid to finish).
  pdl_wait();      // earlier kernels' outputs are visible from here on
  pdl_trigger();
  const int num_tiles = args.identity_T ? (args.identity_T + BN - 1) / BN : *args.num_tiles;
  const int total = num_tiles * nfe;   // a CTA past it publishes no item and only tears down

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_normal();
    const uint64_t pol_x = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    int armed = 0;  // stages armed and not yet known consumed (for the abort path)
    bool ok = true;
    // Items: the CTA's own index first, then from the tile counter
    // (whichever CTA is free takes the next tile) or, without one, every
    // units-th.  Lane 0 fetches one item ahead (the counter's round trip
    // overlaps the current item's loads) and publishes item n + 1 to the
    // ring after the first stage of item n.
    int fetched = 0;
    auto fetch = [&]() -> int {   // the CTA's first item is its own index; the counter hands out the rest
      const int k = fetched++;
      if (k == 0) return unit0;
      return args.next_item ? units + atomicAdd(args.next_item, 1) : unit0 + k * units;
    };
    auto publish = [&](int n, const ItemSlot& v) -> bool {
      const int slot = n & (kItemRing - 1);
      if (!mbar_wait(iempty0 + 8 * slot, ((n / kItemRing) & 1) ^ 1u, &s_abort, wlim)) return false;
      s_ring[slot] = v;
      mbar_arrive(ifull0 + 8 * slot);
      return true;
    };
    ItemSlot cur{}, next{};
    int nxt = -1, got = 1;
    if (lane == 0) {
      cur = slot_of<BN>(args, fetch(), total, num_tiles, nfe);
      got = publish(0, cur) ? 1 : 0;
      if (cur.item >= 0) nxt = fetch();
    }
    if (!__shfl_sync(0xffffffffu, got, 0)) ok = false;
    cur = shfl_slot(cur);
    for (int n = 0; ok && cur.item >= 0; ++n) {
      const int wrow0 = cur.expert * args.w_rows_per_e;
      const int fcol = cur.f * kTileFeat;
      // A tile with at most 32 rows holding routes (decode) loads a 32-row
      // token box and runs N = 32 MMAs (columns of an MMA are independent:
      // each token column's sum over K runs in the same order for any N).
      const bool small = cur.valid <= kSmallRows;
      const int b_rows = small ? kSmallRows : BN;
      const uint32_t stage_tx = C::kABytes + b_rows * kBK * 2;
      for (int ks = 0; ks < ksteps; ++ks) {
        // one lane waits, the warp follows its verdict (keeps the warp converged)
        int got = 1;
        if (lane == 0) got = mbar_wait(empty0 + 8 * stage, phase ^ 1u, &s_abort, wlim) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        uint8_t* sA = smem + stage * C::kStageBytes;
        uint8_t* sB = sA + C::kABytes;
        const uint32_t fb = full0 + 8 * stage;
        const int k0 = ks * kBK;
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, stage_tx);
          tma_load_2d(smem_u32(sA), &w_map, fcol, wrow0 + k0, fb, pol_w);
          tma_load_2d(smem_u32(sA + kBoxBytes), &w_map, fcol + 64, wrow0 + k0, fb, pol_w);
          if (kW13) {
            tma_load_2d(smem_u32(sA + 2 * kBoxBytes), &w_map, args.up_col + fcol, wrow0 + k0, fb, pol_w);
            tma_load_2d(smem_u32(sA + 3 * kBoxBytes), &w_map, args.up_col + fcol + 64, wrow0 + k0, fb, pol_w);
          }
          tma_load_2d(smem_u32(sB), small ? &x_map_small : &x_map, k0, cur.row0, fb, pol_x);
        }
        __syncwarp();
        armed = min(armed + 1, C::kStages);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (ks == 0) {
          int pub = 1;
          if (lane == 0) {
            next = slot_of<BN>(args, nxt, total, num_tiles, nfe);
            pub = publish(n + 1, next) ? 1 : 0;
            if (pub && next.item >= 0) nxt = fetch();
          }
          if (!__shfl_sync(0xffffffffu, pub, 0)) {
            ok = false;
            break;
          }
        }
      }
      cur = shfl_slot(next);
    }
    if (!ok) {
      s_abort = 1;
      if (lane == 0) atomicOr(args.status, kDevErrTimeout);
    }
    if (s_abort && lane == 0) {
      // Let the copies already issued into shared memory land before exit:
      // wait (bounded) for the last `armed` stages' full barriers.
      volatile int no_abort = 0;
      int s = stage;
      uint32_t ph = phase;
      for (int i = 0; i < armed; ++i) {
        if (--s < 0) {
          s = C::kStages - 1;
          ph ^= 1u;
        }
        mbar_wait(full0 + 8 * s, ph, &no_abort);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      // The MMA issue must keep up with the tensor pipe (an M = 128 x N = 128
      // MMA takes ~64 cycles), so the descriptors are built once: those of
      // stage 0 and K step 0, to which a stage adds kStageBytes and a K = 16
      // step 2 KB (A) or 32 B (B) in the 16-byte units of the start-address
      // field.  A: MN-major, 64-feature atoms 8 KB apart (LBO), 8-row K
      // groups 1 KB apart (SBO); B: K-major rows of 128 B.
      const uint64_t adesc0 = sdesc_sw128(smem_u32(smem), kBoxBytes, 1024);
      const uint64_t bdesc0 = sdesc_sw128(smem_u32(smem) + C::kABytes, 16, 1024);
      constexpr uint32_t kStageUnits = C::kStageBytes >> 4;
      uint32_t soff = 0;   // stage * kStageUnits
      for (int n = 0; ok; ++n) {
        const int slot = n & (kItemRing - 1);
        if (!mbar_wait(ifull0 + 8 * slot, (n / kItemRing) & 1, &s_abort, wlim)) {
          ok = false;
          break;
        }
        const ItemSlot it = s_ring[slot];
        mbar_arrive(iempty0 + 8 * slot);
        if (it.item < 0) break;
        const bool small = it.valid <= kSmallRows;
        const uint32_t idesc = small ? C::kIdescSmall : C::kIdesc;
        if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1u, &s_abort, wlim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem + acc * C::kAccCols;
        for (int ks = 0; ks < ksteps; ++ks) {
          if (!mbar_wait(full0 + 8 * stage, phase, &s_abort, wlim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = adesc0 + soff, bd = bdesc0 + soff;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t accum = (ks | kk) != 0 ? 1u : 0u;
            mma_bf16(d0, ad + kk * 128, bd + kk * 2, idesc, accum);
            if (kW13) mma_bf16(d0 + BN, ad + ((2 * kBoxBytes) >> 4) + kk * 128, bd + kk * 2, idesc, accum);
          }
          mma_commit(empty0 + 8 * stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
            soff = 0;
          } else {
            soff += kStageUnits;
          }
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * acc);
        if (++acc == C::kNumAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        s_abort = 1;
        atomicOr(args.status, kDevErrTimeout);
      }
      // all issued MMAs must be complete before TMEM is released
      mma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int feat_local = quarter * 32 + lane;
    const int col0 = ((warp - 2) / 4) * (BN / 2), col1 = col0 + BN / 2;  // this warp's column half
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int n = 0;; ++n) {
      ItemSlot it{};
      it.item = -1;
      int got = 1;
      if (lane == 0) {
        const int slot = n & (kItemRing - 1);
        got = mbar_wait(ifull0 + 8 * slot, (n / kItemRing) & 1, &s_abort, wlim) ? 1 : 0;
        if (got) {
          it = s_ring[slot];
          mbar_arrive(iempty0 + 8 * slot);
        }
      }
      got = __shfl_sync(0xffffffffu, got, 0);
      it = shfl_slot(it);
      if (got && it.item < 0) break;
      TileInfo t{};
      t.row0 = it.row0;
      t.valid = it.valid;
      const int f = it.f;
      if (got && lane == 0) got = mbar_wait(tfull0 + 8 * acc, acc_phase, &s_abort, wlim) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        if (lane == 0) {
          s_abort = 1;
          atomicOr(args.status, kDevErrTimeout);
        }
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + acc * C::kAccCols;
      const int feat = f * kTileFeat + feat_local;
      for (int c = col0; c < col1 && c < t.valid; c += 16) {
        float g[16];
        tmem_ld16(tbase + c, g);
        if (kW13) {
          float u[16];
          tmem_ld16(tbase + BN + c, u);
          tmem_wait_ld();
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int j = c + jj;
            if (j < t.valid) {   // padding rows are not stored: nothing reads them
              const float x = g[jj];
              const float v = __fdividef(x, 1.0f + __expf(-x)) * u[jj];
              out[(size_t)(t.row0 + j) * args.out_ld + feat] = __float2bfloat16_rn(v);
            }
          }
        } else if (args.out_bf16) {
          tmem_wait_ld();
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int j = c + jj;
            if (j < t.valid) out[(size_t)(t.row0 + j) * args.out_ld + feat] = __float2bfloat16_rn(g[jj]);
          }
        } else {
          tmem_wait_ld();
          float* out = reinterpret_cast<float*>(args.out);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int j = c + jj;
            if (j < t.valid) out[(size_t)(t.row0 + j) * args.out_ld + feat] = g[jj];
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty0 + 8 * acc);
      if (++acc == C::kNumAcc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

// ------------------------------------------------------------------ CTA pairs
// The same GEMMs on pairs of CTAs (a cluster of two, one per SM) whose tensor
// cores run one cta_group::2 MMA of M = 256 rows x N = 256 token rows: each
// CTA loads its own 128 rows of the weight tile and half of the token tile
// (128 rows), and its TMEM receives its 128 rows of the result for all 256
// tokens.  Per SM this halves the token bytes per flop, the operand traffic
// that bounds the one-CTA kernel, and keeps both accumulators of a CTA
// (2 x 256 TMEM columns) so that the epilogue of one tile overlaps the MMAs
// of the next.
//   W2 : a CTA's 128 rows are 128 output features (a pair tile: 256).
//   W13: a CTA's 128 rows are 64 gate features followed by the same 64 up
//        features (a pair tile: 128 features).  TMEM lanes 0..63 hold g,
//        lanes 64..127 u; the epilogue warps of lane quarters 2 and 3 pass u
//        through shared memory to the warps of quarters 0 and 1, which store
//        a = silu(g) * u.
// One weight tile shape and one K order (from 0 to the end, 64 per stage, 16
// per MMA) for every tile and every batch.  The MMA's N (token columns) is
// 256, or 64 for a tile with at most 32 routed rows (decode): the columns of
// an MMA are independent dot products over the same K steps, so a token row's
// arithmetic does not depend on the batch, on N, or on which half of the
// tile holds it (the GPU batch-invariance tests compare rows computed with
// N = 64 against the same rows computed with N = 256, bit for bit).
//
// Synchronisation: the even CTA's producer expects the bytes of both CTAs on
// its full barrier, and both CTAs' TMA loads complete there; the even CTA's
// MMA thread commits to the empty and tmem_full barriers of both CTAs; the
// epilogue warps of both CTAs arrive on the even CTA's tmem_empty.  Every
// wait is bounded, and both CTAs of a pair follow the same control flow up to
// the final cluster barrier.
constexpr int kPairRows = 256;      // token rows per pair tile (the MMA's N)
constexpr int kPairM = 256;         // weight rows per pair (the MMA's M)

// kWide (W2 with a long reduction): a work item covers two 256-feature
// groups, two pair MMAs per K step on the same token tile (each the same
// M = 256 x N MMA as one plain item, so the same bits).  Per CTA 48 KB of
// operands per K step for twice the flops: tensor-bound where the plain
// item is bound by the operand bytes an SM takes in; its single
// 512-column accumulator costs the overlap of the epilogue, a few per cent
// of a 14336-deep reduction.
// kDecode (batches of at most 32 tokens, whose tiles all have at most
// kSmallRows routed rows): a stage holds the weight boxes and a kSmallRows-row
// token box, so 9 (W13) or 11 (W2) stages fit instead of 6 or 7.  The MMAs
// are those of a small tile in the other instances (same bits).
template <bool kW13, bool kWide = false, bool kDecode = false>
struct PairCfg {
  static_assert(!(kW13 && kWide), "wide items are W2 only");
  static_assert(!(kWide && kDecode), "decode instances have plain items");
  static constexpr int kGroups = kWide ? 2 : 1;              // 256-feature groups per item
  static constexpr int kRowsCta = kPairRows / 2;
  static constexpr int kFeatCta = kW13 ? 64 : 128;           // output features per CTA and group
  static constexpr int kFeatTile = 2 * kFeatCta * kGroups;   // output features per pair tile
  static constexpr uint32_t kABytes = 2 * kBoxBytes * kGroups;   // 128 weight rows x 64 K per group
  static constexpr uint32_t kBTileBytes = (kDecode ? kSmallRows : kRowsCta) * kBK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBTileBytes;
  // W2 fits a seventh 32 KB stage in the 227 KB of shared memory; W13 needs
  // 16 KB for the u exchange
  static constexpr uint32_t kPairBudget = kW13 ? kStageBudget : 224 * 1024;
  static constexpr int kMaxStages = kDecode ? 12 : 7;
  static constexpr int kStages =
      (int)(kPairBudget / kStageBytes) < kMaxStages ? (int)(kPairBudget / kStageBytes) : kMaxStages;
  static constexpr uint32_t kAccCols = kPairRows * kGroups;
  static constexpr int kNumAcc = kWide ? 1 : 2;
  static constexpr uint32_t kTmemCols = 512;
  // W13: u handed from the up warps to the gate warps, 4 warp pairs x 2
  // buffers x 32 lanes x 16 fp32
  static constexpr uint32_t kXchgBytes = kW13 ? 4 * 2 * 32 * 16 * 4 : 0;
  static constexpr uint32_t kBarBytes = 256;
  static constexpr uint32_t kSmemBytes = kStages * kStageBytes + kXchgBytes + kBarBytes + 1024;
  static constexpr uint32_t kIdesc = idesc_bf16(kPairM, kPairRows, true, false);
  // tiles with at most kSmallRows routed rows: N = 2 x kSmallRows (each CTA
  // supplies kSmallRows token rows)
  static constexpr uint32_t kIdescSmall = idesc_bf16(kPairM, 2 * kSmallRows, true, false);
};

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also returns the AND of `pred` over its threads.
__device__ __forceinline__ int named_bar_and(int id, int threads, int pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred q, p;\n\t"
      "setp.ne.b32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(pred), "r"(id), "r"(threads)
      : "memory");
  return (int)r;
}

template <bool kW13, bool kWide = false, bool kDecode = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    expert_gemm_pair_kernel(const __grid_constant__ CUtensorMap w_map,
                            const __grid_constant__ CUtensorMap x_map,
                            const __grid_constant__ CUtensorMap x_map_small, const GemmArgs args) {
  using C = PairCfg<kW13, kWide, kDecode>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem_base;
  __shared__ volatile int s_abort;

  const uint32_t rank = cluster_ctarank();            // 0: issues the MMAs
  const bool lead = rank == 0;
  const int nfe = args.n_feat_tiles;                  // pair feature tiles (C::kFeatTile features)
  const int pair0 = (int)(blockIdx.x >> 1);
  const int pairs = (int)(gridDim.x >> 1);

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* xchg = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes + C::kXchgBytes);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * C::kStages;
  const uint32_t tfull0 = empty0 + 8 * C::kStages;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ksteps = args.K / kBK;
  const uint64_t wlim = args.wait_ns ? args.wait_ns : kWaitLimitNs;   // pipeline waits

  if (threadIdx.x == 0) {
    for (int st = 0; st < C::kStages; ++st) {
      mbar_init(full0 + 8 * st, 1);
      mbar_init(empty0 + 8 * st, 1);
    }
    for (int b = 0; b < C::kNumAcc; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, 2 * kEpiWarps);   // one arrival per epilogue warp of each CTA
    }
    mbar_init(drain, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&s_tmem_base), C::kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&w_map);
    prefetch_tmap(&x_map);
    prefetch_tmap(&x_map_small);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem = s_tmem_base;
  // The set-up above reads nothing an earlier kernel writes: it overlaps the
  // end of that kernel.  Every CTA of this persistent grid is resident, so
  // the next kernel may launch now (its CTAs wait for this grid to finish).
  pdl_wait();      // earlier kernels' outputs are visible from here on
  pdl_trigger();
  const int num_tiles = args.identity_T ? (args.identity_T + kPairRows - 1) / kPairRows : *args.num_tiles;
  const int total = num_tiles * nfe;   // a pair past it runs no item and only tears down

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    const uint64_t pol_w = policy_evict_normal();
    const uint64_t pol_x = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    int armed = 0;
    bool ok = true;
    for (int item = pair0; item < total && ok; item += pairs) {
      const Work wk = work_of<kPairRows>(args, item, num_tiles, nfe);
      const TileInfo t = wk.t;
      const int wrow0 = t.expert * args.w_rows_per_e;
      const int fcol = wk.f * C::kFeatTile + (int)rank * C::kFeatCta;   // this CTA's features (group 0)
      // tiles with at most kSmallRows routed rows (decode): a kSmallRows-row
      // token box per CTA and N = 2 kSmallRows MMAs; the odd CTA's rows are
      // padding or beyond the tile, in columns that are never stored
      const bool small = kDecode || t.valid <= kSmallRows;
      // (a decode instance given a tile of more rows computes only its first
      // kSmallRows: reported, never silent)
      if (kDecode && t.valid > kSmallRows && lane == 0) atomicOr(args.status, kDevErrBadBlocks);
      const int b_rows = small ? kSmallRows : C::kRowsCta;
      const int brow0 = t.row0 + (int)rank * b_rows;                     // this CTA's half of the rows
      const uint32_t cta_tx = C::kABytes + b_rows * kBK * 2;
      for (int ks = 0; ks < ksteps; ++ks) {
        int got = 1;
        if (lane == 0) got = mbar_wait_cluster(empty0 + 8 * stage, phase ^ 1u, &s_abort, wlim) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        uint8_t* sA = smem + stage * C::kStageBytes;
        uint8_t* sB = sA + C::kABytes;
        const uint32_t fb = mapa_shared(full0 + 8 * stage, 0);   // the even CTA's full barrier
        const int k0 = ks * kBK;
        if (lane == 0) {
          if (lead) mbar_arrive_expect_tx(full0 + 8 * stage, 2 * cta_tx);
          // rows 0..63 and 64..127 of this CTA's weight tile: two 64-wide boxes
          const int c_hi = kW13 ? args.up_col + fcol : fcol + 64;
          tma_load_2d_pair(smem_u32(sA), &w_map, fcol, wrow0 + k0, fb, pol_w);
          tma_load_2d_pair(smem_u32(sA + kBoxBytes), &w_map, c_hi, wrow0 + k0, fb, pol_w);
          if (kWide) {   // group 1: the next 256 features of the item
            tma_load_2d_pair(smem_u32(sA + 2 * kBoxBytes), &w_map, fcol + 256, wrow0 + k0, fb, pol_w);
            tma_load_2d_pair(smem_u32(sA + 3 * kBoxBytes), &w_map, fcol + 256 + 64, wrow0 + k0, fb, pol_w);
          }
          tma_load_2d_pair(smem_u32(sB), small ? &x_map_small : &x_map, k0, brow0, fb, pol_x);
        }
        __syncwarp();
        armed = min(armed + 1, C::kStages);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok) {
      s_abort = 1;
      if (lane == 0) atomicOr(args.status, kDevErrTimeout);
    }
    if (s_abort && lane == 0) {
      if (lead) {
        // copies already issued (ours and the odd CTA's) complete on our full
        // barriers: let them land before exit
        volatile int no_abort = 0;
        int st = stage;
        uint32_t ph = phase;
        for (int i = 0; i < armed; ++i) {
          if (--st < 0) {
            st = C::kStages - 1;
            ph ^= 1u;
          }
          mbar_wait_cluster(full0 + 8 * st, ph, &no_abort);
        }
      } else {
        // the odd CTA's copies complete on the even CTA's barriers: give any
        // still in flight time to land in our shared memory
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 200000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lead && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      // descriptors built once (see the one-CTA kernel); a stage adds
      // kStageBytes, a K = 16 step 2 KB (A) or 32 B (B), wide items' second
      // group 16 KB (A)
      const uint64_t adesc0 = sdesc_sw128(smem_u32(smem), kBoxBytes, 1024);
      const uint64_t bdesc0 = sdesc_sw128(smem_u32(smem) + C::kABytes, 16, 1024);
      constexpr uint32_t kStageUnits = C::kStageBytes >> 4;
      uint32_t soff = 0;   // stage * kStageUnits
      // the routed rows of the next item's tile are loaded one item ahead
      int valid = pair0 < total ? work_of<kPairRows>(args, pair0, num_tiles, nfe).t.valid : 0;
      for (int item = pair0; item < total && ok; item += pairs) {
        const bool small = kDecode || valid <= kSmallRows;
        const uint32_t idesc = small ? C::kIdescSmall : C::kIdesc;
        valid = item + pairs < total ? work_of<kPairRows>(args, item + pairs, num_tiles, nfe).t.valid : 0;
        if (!mbar_wait_cluster(tempty0 + 8 * acc, acc_phase ^ 1u, &s_abort, wlim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem + acc * C::kAccCols;
        for (int ks = 0; ks < ksteps; ++ks) {
          if (!mbar_wait_cluster(full0 + 8 * stage, phase, &s_abort, wlim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = adesc0 + soff, bd = bdesc0 + soff;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t accum = (ks | kk) != 0 ? 1u : 0u;
            mma_bf16_pair(d0, ad + kk * 128, bd + kk * 2, idesc, accum);
            if (kWide) mma_bf16_pair(d0 + kPairRows, ad + ((2 * kBoxBytes) >> 4) + kk * 128, bd + kk * 2, idesc, accum);
          }
          mma_commit_pair(empty0 + 8 * stage, 0x3);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
            soff = 0;
          } else {
            soff += kStageUnits;
          }
        }
        if (!ok) break;
        mma_commit_pair(tfull0 + 8 * acc, 0x3);
        if (++acc == C::kNumAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        s_abort = 1;
        atomicOr(args.status, kDevErrTimeout);
      }
      mma_commit_pair(drain, 0x1);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int quarter = warp & 3;                       // TMEM lanes this warp may access
    const int half = (warp - 2) / 4;                    // its half of the 256 columns
    const int col0 = half * (kPairRows / 2), col1 = col0 + kPairRows / 2;
    // W13: quarters 0,1 hold g (features 0..63 of the CTA), quarters 2,3 hold u
    const bool up_warp = kW13 && quarter >= 2;
    const int xpair = (quarter & 1) + 2 * half;         // W13: the (gate, up) warp pair
    float* xbuf = xchg + (size_t)xpair * 2 * 32 * 16;   // two buffers of 32 lanes x 16
    int acc = 0;
    uint32_t acc_phase = 0;
    int chunk = 0;                                      // W13: exchange buffer parity
    for (int item = pair0; item < total; item += pairs) {
      const Work wk = work_of<kPairRows>(args, item, num_tiles, nfe);
      const TileInfo t = wk.t;
      int got = 1;
      if (lane == 0) got = mbar_wait_cluster(tfull0 + 8 * acc, acc_phase, &s_abort, wlim) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
      // W13: the gate and up warps of a pair meet on a named barrier for
      // every chunk of the tile, so they take the same verdict (one of them
      // must not go on to the exchange while the other gives up)
      if (kW13) got = named_bar_and(1 + xpair, 64, got);
      if (!got) {
        if (lane == 0) {
          s_abort = 1;
          atomicOr(args.status, kDevErrTimeout);
        }
        break;
      }
      tc_fence_after();
      for (int grp = 0; grp < C::kGroups; ++grp) {
      const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + acc * C::kAccCols + grp * kPairRows;
      const int feat = wk.f * C::kFeatTile + grp * 256 + (int)rank * C::kFeatCta +
                       (kW13 ? (quarter & 1) * 32 : quarter * 32) + lane;
      for (int c = col0; c < col1 && c < t.valid; c += 16) {
        float v[16];
        tmem_ld16(tbase + c, v);
        tmem_wait_ld();
        if (kW13) {
          // [column][lane] order: the 32 lanes touch 32 consecutive words
          float* buf = xbuf + (chunk & 1) * (32 * 16) + lane;
          if (up_warp) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) buf[jj * 32] = v[jj];
            named_bar_sync(1 + xpair, 64);
          } else {
            named_bar_sync(1 + xpair, 64);
            __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int j = c + jj;
              if (j < t.valid) {   // padding rows are not stored: nothing reads them
                const float x = v[jj];
                const float a = __fdividef(x, 1.0f + __expf(-x)) * buf[jj * 32];
                out[(size_t)(t.row0 + j) * args.out_ld + feat] = __float2bfloat16_rn(a);
              }
            }
          }
          ++chunk;
        } else if (args.out_bf16) {
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int j = c + jj;
            if (j < t.valid) out[(size_t)(t.row0 + j) * args.out_ld + feat] = __float2bfloat16_rn(v[jj]);
          }
        } else {
          float* out = reinterpret_cast<float*>(args.out);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int j = c + jj;
            if (j < t.valid) out[(size_t)(t.row0 + j) * args.out_ld + feat] = v[jj];
          }
        }
      }
      }   // groups
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa_shared(tempty0 + 8 * acc, 0));
      if (++acc == C::kNumAcc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // nothing of either CTA still targets the other's shared memory
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, C::kTmemCols);
}

template <bool kW13, int BN>
void launch(const CUtensorMap& w_map, const CUtensorMap& x_map, const CUtensorMap& x_small,
            GemmArgs a, int max_tiles, int num_sms, cudaStream_t s) {
  auto kernel = expert_gemm_kernel<kW13, BN>;
  const int smem = (int)GemmCfg<kW13, BN>::kSmemBytes;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const long long items = (long long)max_tiles * a.n_feat_tiles;
  if (items <= 0) return;
  const int grid = (int)(items < num_sms ? items : num_sms);
  a.concurrent = grid;
  launch_pdl(kernel, dim3(grid), dim3(kThreads), smem, s, w_map, x_map, x_small, a);
}

// Pairs of CTAs that can be resident at once (one CTA per SM; a pair needs
// two SMs of one GPC), looked up once per device and kernel.
template <bool kW13, bool kWide = false, bool kDecode = false>
int resident_pairs(int num_sms) {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (unsigned)(num_sms / 2), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = PairCfg<kW13, kWide, kDecode>::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&n, expert_gemm_pair_kernel<kW13, kWide, kDecode>, &cfg) != cudaSuccess ||
      n <= 0) {
    cudaGetLastError();
    n = num_sms / 2;
  }
  n = n < num_sms / 2 ? n : num_sms / 2;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

template <bool kW13, bool kWide = false, bool kDecode = false>
void launch_pair(const CUtensorMap& w_map, const CUtensorMap& x_map, const CUtensorMap& x_small, GemmArgs a,
                 int max_tiles, int num_sms, cudaStream_t s) {
  auto kernel = expert_gemm_pair_kernel<kW13, kWide, kDecode>;
  const int smem = (int)PairCfg<kW13, kWide, kDecode>::kSmemBytes;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const long long items = (long long)max_tiles * a.n_feat_tiles;
  if (items <= 0) return;
  const int cap = resident_pairs<kW13, kWide, kDecode>(num_sms);
  const int pairs = (int)(items < cap ? items : cap);
  a.concurrent = pairs;
  launch_pdl(kernel, dim3(2 * pairs), dim3(kThreads), smem, s, w_map, x_map, x_small, a);
}

}  // namespace

bool gemm_smem_ok() {
  int dev = 0, optin = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  return optin >= (int)GemmCfg<true, kW13TileRows>::kSmemBytes &&
         optin >= (int)GemmCfg<false, kW2TileRows>::kSmemBytes &&
         optin >= (int)GemmCfg<false, kRouterTileRows>::kSmemBytes &&
         optin >= (int)GemmCfg<false, kRouterTileRowsNarrow>::kSmemBytes &&
         optin >= (int)PairCfg<true>::kSmemBytes && optin >= (int)PairCfg<false>::kSmemBytes &&
         optin >= (int)PairCfg<false, true>::kSmemBytes &&
         optin >= (int)PairCfg<true, false, true>::kSmemBytes &&
         optin >= (int)PairCfg<false, false, true>::kSmemBytes;
}

bool gemm_pair_ok(bool w13, int features, int K) {
  // (the one-CTA W13, two M = 128 x N = 128 MMAs per K step, measured slower
  // for every reduction length once the MMA issue loop was tight: Qwen-like
  // W13 0.307 against 0.279 ms at K = 2048)
  (void)K;
  return features % (w13 ? PairCfg<true>::kFeatTile : PairCfg<false>::kFeatTile) == 0;
}

bool gemm_wide_ok(int features, int K) {
  return features % PairCfg<false, true>::kFeatTile == 0 && K >= kWideMinK;
}

void launch_w13_gemm(const CUtensorMap& w_map, const CUtensorMap& x_map, const CUtensorMap& x_small,
                     const GemmArgs& a, int max_tiles, int num_sms, cudaStream_t s) {
  if (a.pair && a.decode)
    launch_pair<true, false, true>(w_map, x_map, x_small, a, max_tiles, num_sms, s);
  else if (a.pair)
    launch_pair<true>(w_map, x_map, x_small, a, max_tiles, num_sms, s);
  else
    launch<true, kW13TileRows>(w_map, x_map, x_small, a, max_tiles, num_sms, s);
}

void launch_w2_gemm(const CUtensorMap& w_map, const CUtensorMap& x_map, const CUtensorMap& x_small,
                    const GemmArgs& a, int max_tiles, int num_sms, cudaStream_t s) {
  if (a.pair && a.wide)
    launch_pair<false, true>(w_map, x_map, x_small, a, max_tiles, num_sms, s);
  else if (a.pair && a.decode)
    launch_pair<false, false, true>(w_map, x_map, x_small, a, max_tiles, num_sms, s);
  else if (a.pair)
    launch_pair<false>(w_map, x_map, x_small, a, max_tiles, num_sms, s);
  else
    launch<false, kW2TileRows>(w_map, x_map, x_small, a, max_tiles, num_sms, s);
}

void launch_router_gemm(const CUtensorMap& w_map, const CUtensorMap& x_map, const CUtensorMap& x_small,
                        const GemmArgs& a, int max_tiles, int num_sms, cudaStream_t s, int tile_rows) {
  if (tile_rows == kRouterTileRowsNarrow)
    launch<false, kRouterTileRowsNarrow>(w_map, x_map, x_small, a, max_tiles, num_sms, s);
  else
    launch<false, kRouterTileRows>(w_map, x_map, x_small, a, max_tiles, num_sms, s);
}

}  // namespace moe
