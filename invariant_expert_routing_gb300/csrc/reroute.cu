// Overflow reroute ("Mixture-of-Experts Routing at Inference Time", Figure 2,
// the reroute branch of the overflow policy, and the mitigation after
// routing_stats: overflow goes to the next-choice expert instead of skipping
// the expert tier).
//
// Definition (the sequential rule).  Phase one is the drop policy: route r
// keeps its expert if its rank among that expert's routes is below C.  Phase
// two visits the routes phase one would drop in ascending r; each takes the
// best-ranked expert of its token (larger logit, then lower index, NaN last)
// that still has room and that the token does not use yet (its k chosen
// experts and the targets of its earlier slots), or stays dropped.
//
// Computation.  The sequential rule is a serial dictatorship with one
// priority order (route id) shared by every expert, so deferred acceptance
// computes it in parallel rounds: every unplaced route proposes to its best
// expert that could still take it, and every expert keeps the proposals and
// holders of lowest route id up to its room.  A token's later slot may not
// take an expert an earlier slot of the token holds or proposes to.  The
// rounds run in one CTA (reroute_da_kernel) for small batches and across a
// co-resident grid (reroute_da_grid_kernel) for large ones; proposals walk a
// cached list of each token's best experts (reroute_prefs_kernel), with a
// full scan once the list is used up.  The outcome is then checked against a characterisation of
// the sequential rule (reroute_verify_kernel): every target is usable, and
// every usable expert a route ranks above its outcome is full with routes of
// higher priority.  An assignment that passes is the sequential one (at each
// route's turn its target had room and every better usable expert did not).
// If the check fails or the rounds do not settle, reroute_seq_kernel, a
// direct implementation of the sequential rule, recomputes the assignment.
// Every decision is on integers, so the result is the same bits either way.
#include <cstdint>

#include "kernels.h"

namespace moe {
namespace {

constexpr int kMaxN = 256;
constexpr int kRerouteThreads = 1024;

// Ranking key: larger is better; NaN below every number, -0 equal to +0,
// equal logits ordered by lower expert index.  0 means "no expert".
__device__ __forceinline__ unsigned long long reroute_key(float l, int e) {
  uint32_t key = 0u;
  if (!isnan(l)) {
    uint32_t u = __float_as_uint(l);
    if (u == 0x80000000u) u = 0u;
    key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  return ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)e);
}

__device__ __forceinline__ int key_expert(unsigned long long key) {
  return (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
}

// Phase one for route r: its expert if kept, -1 if it overflows (or has none).
__device__ __forceinline__ bool phase_one_overflow(const int32_t* __restrict__ topk_idx,
                                                   const int32_t* __restrict__ rank_in_tile,
                                                   const int32_t* __restrict__ tile_base, int N,
                                                   int capacity, long long r, int* kept_e) {
  const int e = topk_idx[r];
  *kept_e = -1;
  if (e < 0 || e >= N) return false;
  const int rank = tile_base[(size_t)(r / kDispatchTile) * N + e] + rank_in_tile[r];
  if (rank < capacity) {
    *kept_e = e;
    return false;
  }
  return true;
}

// ---------------------------------------------------------------- preference lists
// Every slot of a token shares one list: the token's experts outside its own
// top-k, best first.  One warp per token that has an overflowing slot; the
// warp sorts the token's N ranking keys (own experts and padding set to 0)
// with a bitonic network, V keys per lane, element i in lane i / V, and keeps
// the first min(L, N - k).
template <int V>
__device__ __forceinline__ void warp_sort_desc(unsigned long long (&a)[V]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32 * V; size <<= 1) {
#pragma unroll
    for (int j = size >> 1; j > 0; j >>= 1) {
      if (j >= V) {   // partner: same slot of lane ^ (j / V)
#pragma unroll
        for (int s = 0; s < V; ++s) {
          const int i = lane * V + s;
          const unsigned long long b = __shfl_xor_sync(0xffffffffu, a[s], j / V);
          const bool keep_max = ((i & j) == 0) == ((i & size) == 0);
          a[s] = keep_max ? (a[s] > b ? a[s] : b) : (a[s] < b ? a[s] : b);
        }
      } else {        // partner: slot s + j of this lane
#pragma unroll
        for (int s = 0; s < V; ++s) {
          if ((s & j) == 0) {
            const bool desc = ((lane * V + s) & size) == 0;
            const unsigned long long x = a[s], y = a[s + j];
            const unsigned long long hi = x > y ? x : y, lo = x > y ? y : x;
            a[s] = desc ? hi : lo;
            a[s + j] = desc ? lo : hi;
          }
        }
      }
    }
  }
}

template <int V>
__global__ void __launch_bounds__(256) reroute_prefs_kernel(
    const int32_t* __restrict__ topk_idx, const float* __restrict__ logits, int T, int N, int k,
    int capacity, const int32_t* __restrict__ rank_in_tile, const int32_t* __restrict__ tile_base,
    int L, uint8_t* __restrict__ prefs, uint32_t* __restrict__ gsync, int32_t* __restrict__ flag) {
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x < 4) {   // barrier state and flag of the rounds that follow
    if (threadIdx.x < 3) gsync[threadIdx.x] = 0u;
    else *flag = 0;
  }
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  bool over = false;
  if (lane < k) {
    int kept_e = -1;
    over = phase_one_overflow(topk_idx, rank_in_tile, tile_base, N, capacity, (long long)t * k + lane,
                              &kept_e);
  }
  if (!__any_sync(0xffffffffu, over)) return;
  unsigned long long key[V];
#pragma unroll
  for (int s = 0; s < V; ++s) {
    const int e = lane * V + s;
    key[s] = e < N ? reroute_key(logits[(size_t)t * N + e], e) : 0ull;
  }
  for (int q = 0; q < k; ++q) {   // the token's own experts are not candidates
    const int e = topk_idx[(long long)t * k + q];
#pragma unroll
    for (int s = 0; s < V; ++s)
      if (e == lane * V + s) key[s] = 0ull;
  }
  warp_sort_desc<V>(key);
  const int n = min(L, N - k);
#pragma unroll
  for (int s = 0; s < V; ++s) {
    const int i = lane * V + s;
    if (i < n) prefs[(size_t)t * L + i] = (uint8_t)key_expert(key[s]);
  }
}

// Block-wide exclusive scan of one int per thread (kRerouteThreads threads).
__device__ int block_scan_1024(int v, int* wbuf, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = v;
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) wbuf[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int c = wbuf[lane];
    int wi = c;
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += y;
    }
    wbuf[lane] = wi - c;
    if (lane == 31) wbuf[32] = wi;
  }
  __syncthreads();
  const int res = wbuf[w] + incl - v;
  *total = wbuf[32];
  __syncthreads();
  return res;
}

// ---------------------------------------------------------------- list walk
// Expert id at position b of a 16-entry window.
__device__ __forceinline__ int window_expert(unsigned long long lo, unsigned long long hi, int b) {
  return (int)(((b < 8 ? lo : hi) >> (8 * (b & 7))) & 0xFFull);
}

// The first position >= p of a token's preference list (length Leff) whose
// expert can still take route r (r < thresh[e]) and is not held by one of the
// token's earlier slots (hold[q0..q1), entries < 0 hold nothing); -1 if none.
// p moves to that position (Leff if none).  Sixteen entries are tested at a
// time; positions below Lc come from the shared-memory copy `cached`, the
// rest from `row` in global memory.
__device__ __forceinline__ int walk_list(const uint8_t* cached, int Lc, const uint8_t* __restrict__ row,
                                         int Leff, int& p, int r, const int* thresh, const int* hold,
                                         int q0, int q1) {
  while (p < Leff) {
    const int base = p & ~15;
    const uint4 v = base < Lc ? *reinterpret_cast<const uint4*>(cached + base)
                              : *reinterpret_cast<const uint4*>(row + base);
    const unsigned long long lo = (unsigned long long)v.x | ((unsigned long long)v.y << 32);
    const unsigned long long hi = (unsigned long long)v.z | ((unsigned long long)v.w << 32);
    unsigned m = 0u;
#pragma unroll
    for (int b = 0; b < 16; ++b) {
      const int e = window_expert(lo, hi, b);
      const bool ok = base + b >= p && base + b < Leff && r < thresh[e];
      m |= (ok ? 1u : 0u) << b;
    }
    while (m) {
      const int b = __ffs(m) - 1;
      const int e = window_expert(lo, hi, b);
      bool ex = false;
      for (int q = q0; q < q1; ++q) ex |= hold[q] == e;
      if (!ex) {
        p = base + b;
        return e;
      }
      m &= m - 1u;
    }
    p = base + 16;
  }
  p = Leff;
  return -1;
}

// ---------------------------------------------------------------- deferred acceptance
// hold[i] (list position i): the expert route list[i] holds, -1 none yet,
// -2 no expert can take it any more.  cnt/worst: after each round, how many
// overflow routes each expert holds and the largest such route id (-1 none);
// an expert can still take route r if cnt < room or worst > r.
__global__ void __launch_bounds__(kRerouteThreads, 1) reroute_da_kernel(
    const int32_t* __restrict__ topk_idx, const float* __restrict__ logits, int T, int N, int k,
    int capacity, const int32_t* __restrict__ rank_in_tile, const int32_t* __restrict__ tile_base,
    const int32_t* __restrict__ kept_count, RerouteScratch sc, int L, int max_rounds,
    int32_t* __restrict__ route_expert, int32_t* __restrict__ num_dropped,
    int32_t* __restrict__ num_rerouted) {
  __shared__ int room[kMaxN], cnt[kMaxN], worst[kMaxN], acc[kMaxN], nworst[kMaxN];
  // thresh[e]: expert e can still take route r iff r < thresh[e] (INT_MAX while it has room)
  __shared__ int thresh[kMaxN];
  __shared__ int tab[32][kMaxN + 1];
  __shared__ int wbuf[33];
  __shared__ int s_unplaced;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const long long R = (long long)T * k;
  const int Leff = min(L, N - k);
  const bool lists_complete = Leff == N - k;
  if (tid == 0) *sc.flag = 0;
  for (int e = tid; e < N; e += blockDim.x) {
    room[e] = capacity - kept_count[e];
    cnt[e] = 0;
    worst[e] = -1;
    thresh[e] = room[e] > 0 ? 0x7FFFFFFF : -1;
  }
  // phase one for every route; the overflowing ones listed in route order
  int M = 0;
  for (long long base = 0; base < R; base += kRerouteThreads) {
    const long long r = base + tid;
    bool over = false;
    if (r < R) {
      int kept_e = -1;
      over = phase_one_overflow(topk_idx, rank_in_tile, tile_base, N, capacity, r, &kept_e);
      route_expert[r] = kept_e;
    }
    int nprev = 0;   // earlier overflowing slots of the same token
    if (over) {
      const long long t0 = (r / k) * k;
      for (long long q = t0; q < r; ++q) {
        int kq = -1;
        nprev += phase_one_overflow(topk_idx, rank_in_tile, tile_base, N, capacity, q, &kq) ? 1 : 0;
      }
    }
    int total = 0;
    const int pos = block_scan_1024(over ? 1 : 0, wbuf, &total);
    if (over) {
      sc.list[M + pos] = (int32_t)r;
      sc.hold[M + pos] = -1;
      sc.ptr[M + pos] = 0;
      sc.first[M + pos] = M + pos - nprev;
    }
    M += total;
  }
  __syncthreads();
  bool settled = M == 0;
  for (int round = 0; round < max_rounds && !settled; ++round) {
    // (a) proposals of the unplaced routes, from the previous round's state
    for (int i0 = 0; i0 < M; i0 += kRerouteThreads) {
      const int i = i0 + tid;
      if (i >= M) continue;
      const int h = sc.hold[i];
      if (h != -1) {
        sc.cand[i] = h;
        continue;
      }
      const int r = sc.list[i];
      const int t = r / k;
      const int f = sc.first[i];   // the token's earlier overflowing slots: f .. i-1
      int p = sc.ptr[i];
      int chosen = walk_list(nullptr, 0, sc.prefs + (size_t)t * L, Leff, p, r, thresh, sc.hold, f, i);
      sc.ptr[i] = p;
      if (chosen < 0 && !lists_complete) {
        // the cached list is used up: scan every expert
        uint32_t own[kMaxN / 32];
        for (int x = 0; x < kMaxN / 32; ++x) own[x] = 0u;
        for (int q = 0; q < k; ++q) {
          const int e1 = topk_idx[(long long)t * k + q];
          if (e1 >= 0 && e1 < N) own[e1 >> 5] |= 1u << (e1 & 31);
        }
        for (int q = f; q < i; ++q) {
          const int hq = sc.hold[q];
          if (hq >= 0) own[hq >> 5] |= 1u << (hq & 31);
        }
        unsigned long long best = 0ull;
        for (int e = 0; e < N; ++e) {
          if (((own[e >> 5] >> (e & 31)) & 1u) || !(r < thresh[e])) continue;
          const unsigned long long key = reroute_key(logits[(size_t)t * N + e], e);
          best = key > best ? key : best;
        }
        if (best) chosen = key_expert(best);
      }
      sc.cand[i] = chosen >= 0 ? chosen : -2;
    }
    for (int e = tid; e < N; e += blockDim.x) {
      acc[e] = 0;
      nworst[e] = -1;
    }
    if (tid == 0) s_unplaced = 0;
    __syncthreads();
    // (b) every expert keeps its candidates of lowest route id, up to its room
    for (int i0 = 0; i0 < M; i0 += kRerouteThreads) {
      const int i = i0 + tid;
      int c = -1, r = 0;
      if (i < M) {
        c = sc.cand[i];
        r = sc.list[i];
        if (c >= 0)   // a token's later slot yields to an earlier slot's candidate
          for (int q = sc.first[i]; q < i; ++q)
            if (sc.cand[q] == c) c = -1;
      }
      for (int x = tid; x < 32 * (kMaxN + 1); x += blockDim.x) (&tab[0][0])[x] = 0;
      __syncthreads();
      const int key = c >= 0 ? c : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      const int wrank = __popc(peers & ((1u << lane) - 1u));
      if (c >= 0 && wrank == 0) tab[w][c] = __popc(peers);
      __syncthreads();
      for (int e = tid; e < N; e += blockDim.x) {
        int run = acc[e];
        for (int ww = 0; ww < 32; ++ww) {
          const int v = tab[ww][e];
          tab[ww][e] = run;
          run += v;
        }
        acc[e] = run;
      }
      __syncthreads();
      if (i < M) {
        int nh;
        if (c >= 0 && tab[w][c] + wrank < room[c]) {
          nh = c;
          atomicMax(&nworst[c], r);
        } else {
          nh = sc.cand[i] == -2 ? -2 : -1;
        }
        sc.hold[i] = nh;
        route_expert[r] = nh >= 0 ? nh : -1;
        if (nh == -1) s_unplaced = 1;
      }
      __syncthreads();
    }
    for (int e = tid; e < N; e += blockDim.x) {
      cnt[e] = min(acc[e], room[e]);
      worst[e] = nworst[e];
      thresh[e] = cnt[e] < room[e] ? 0x7FFFFFFF : worst[e];
    }
    __syncthreads();
    settled = s_unplaced == 0;
    __syncthreads();
  }
  // results: counts of rerouted and still dropped routes, expert state
  int rer = 0, drop = 0;
  for (int i = tid; i < M; i += blockDim.x) {
    if (sc.hold[i] >= 0) ++rer;
    else ++drop;
  }
  int tr = 0, td = 0;
  block_scan_1024(rer, wbuf, &tr);
  block_scan_1024(drop, wbuf, &td);
  for (int e = tid; e < N; e += blockDim.x) {
    sc.acc[e] = cnt[e];
    sc.worst[e] = worst[e];
  }
  if (tid == 0) {
    *num_rerouted = tr;
    *num_dropped = td;
    *sc.count = M;
    if (!settled) *sc.flag = 1;
  }
}

// ---------------------------------------------------------------- grid-wide deferred acceptance
// The same rounds as reroute_da_kernel, spread over a co-resident grid
// (cooperative launch, one CTA per SM) for batches with many overflowing
// routes.  CTA X owns the routes [X*S, X*S + S), S a multiple of k, so the
// slots of a token never span two CTAs: the CTA keeps its overflowing routes
// (route id, holding, list position, first slot of the token, candidate,
// rank) in shared memory for the whole pass.  A round:
//   (a) every unplaced route of the CTA proposes (its best expert that could
//       still take it, the token's held experts excluded);
//   (b) a later slot yields to an earlier slot's candidate; each candidate's
//       rank among the CTA's candidates of its expert; the CTA publishes its
//       per-expert counts (16-bit, expert-major), their exclusive prefix over
//       experts, the number of routes no expert can take, the number of
//       listed routes, and its candidates' route ids ordered by (expert, rank);
//   -- device-wide barrier --
//   (c) every CTA copies all CTAs' counts into shared memory (cp.async, one
//       round trip) and derives each expert's total, this CTA's prefix (its
//       candidates' global ranks: lowest route ids win, since CTAs own
//       ascending route ranges) and where the expert's last accepted
//       candidate sits; two dependent loads fetch that route id (the
//       threshold of the next round).  The number of still unplaced routes
//       follows from the totals, so every CTA takes the same decision to stop.
// The published arrays alternate between two buffers by round, so a buffer
// is rewritten only after every CTA has passed the next barrier.  Data that
// other CTAs write is read with ld.global.cg (L2), as L1 is not coherent
// across SMs.  A barrier that waits longer than its limit (kBarrierLimitNs
// unless the caller passes a shorter one) records an error: every CTA then
// leaves at its next barrier, and the flag hands the batch to the sequential
// kernel.
constexpr unsigned long long kBarrierLimitNs = 200000000ull;   // 0.2 s
constexpr int kGridMaxChunks = 3;   // 1024-route chunks per CTA (24 KB of shared memory each)

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// gs[0] counts arrivals over the whole launch: the b-th barrier (from 0) is
// passed once it reaches G * (b + 1) (at most 152 CTAs x 1040 rounds, far
// below 2^30).  A CTA that gives up sets bit 30 (an OR, so that several CTAs
// giving up at once cannot carry it away), which releases every waiter and
// marks the error.  Uniform result in the CTA.
constexpr uint32_t kBarrierError = 1u << 30;

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ bool grid_barrier(uint32_t* gs, uint32_t target, int* s_ok, unsigned long long limit_ns) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(&gs[0], 1u);
    uint32_t v = ld_acquire_gpu(&gs[0]);
    if (v < target) {
      const unsigned long long t0 = global_ns();
      while ((v = ld_acquire_gpu(&gs[0])) < target) {
        if (global_ns() - t0 > limit_ns) {
          atomicOr(&gs[0], kBarrierError);
          v = kBarrierError;
          break;
        }
      }
    }
    __threadfence();
    *s_ok = v < kBarrierError ? 1 : 0;
  }
  __syncthreads();
  return *s_ok != 0;
}

// Block-wide sum of one int per thread (kRerouteThreads threads).
__device__ __forceinline__ int block_sum_1024(int v, int* wbuf) {
  int total = 0;
  block_scan_1024(v, wbuf, &total);
  return total;
}

// Lanes of the warp whose expert equals this lane's (c >= 0), from one ballot
// per bit of the expert id; meaningful only where c >= 0.
__device__ __forceinline__ unsigned lanes_with_expert(int c, int bits) {
  unsigned m = __ballot_sync(0xffffffffu, c >= 0);
  for (int b = 0; b < bits; ++b) {
    const bool on = (c >> b) & 1;
    const unsigned bl = __ballot_sync(0xffffffffu, on);
    m &= on ? bl : ~bl;
  }
  return m;
}

__device__ __forceinline__ void cp_async_16(void* smem, const void* gmem) {
  const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__global__ void __launch_bounds__(kRerouteThreads, 1) reroute_da_grid_kernel(
    const int32_t* __restrict__ topk_idx, const float* __restrict__ logits, int T, int N, int k,
    int capacity, const int32_t* __restrict__ rank_in_tile, const int32_t* __restrict__ tile_base,
    const int32_t* __restrict__ kept_count, RerouteScratch sc, int L, int Lc, int max_rounds, int S,
    int chunks, int32_t* __restrict__ route_expert, int32_t* __restrict__ num_dropped,
    int32_t* __restrict__ num_rerouted, unsigned long long barrier_ns, int* __restrict__ status) {
  extern __shared__ __align__(16) int dyn[];
  const int cap = chunks * kRerouteThreads;
  int* e_r = dyn;
  int* e_hold = dyn + cap;
  int* e_ptr = dyn + 2 * cap;
  int* e_first = dyn + 3 * cap;
  int* e_cand = dyn + 4 * cap;
  int* e_rank = dyn + 5 * cap;
  uint16_t* stage = reinterpret_cast<uint16_t*>(dyn + 6 * cap);   // [N + 2][gs] counts of every CTA
  __shared__ int room[kMaxN], thresh[kMaxN], cnt[kMaxN], off[kMaxN], worst[kMaxN];
  __shared__ int pre[kMaxN + 2], tot[kMaxN + 2], cross_x[kMaxN], cross_q[kMaxN];
  __shared__ int part[kRerouteThreads];
  __shared__ int tab[32][kMaxN + 1];
  __shared__ int wbuf[33];
  __shared__ int s_ok;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int X = blockIdx.x, G = gridDim.x;
  const int gs = (G + 7) / 8 * 8;
  const size_t xints = reroute_exchange_ints(G, N);
  // the first Lc entries of the lists of this CTA's tokens
  uint8_t* pcache = reinterpret_cast<uint8_t*>(stage + (size_t)(N + 2) * gs);
  const long long R = (long long)T * k;
  const long long r0 = (long long)X * S;
  const long long r1 = min(R, r0 + (long long)S);
  const int Leff = min(L, N - k);
  const bool lists_complete = Leff == N - k;
  const int t0 = (int)(r0 / k);
  for (int e = tid; e < N; e += blockDim.x) {
    room[e] = capacity - kept_count[e];
    thresh[e] = room[e] > 0 ? 0x7FFFFFFF : -1;
  }
  {
    const int ntok = (int)((r1 - r0) / k), per_row = Lc / 16;
    for (int c = tid; c < ntok * per_row; c += blockDim.x) {
      const int tt = c / per_row, q = c % per_row;
      cp_async_16(pcache + (size_t)tt * Lc + 16 * q, sc.prefs + (size_t)(t0 + tt) * L + 16 * q);
    }
    cp_async_wait_all();
  }
  // phase one over this CTA's routes; the overflowing ones listed in route order
  int n = 0;
  for (long long base = r0; base < r1; base += kRerouteThreads) {
    const long long r = base + tid;
    bool over = false;
    int nprev = 0;   // earlier overflowing slots of the same token
    if (r < r1) {
      int kept_e = -1;
      over = phase_one_overflow(topk_idx, rank_in_tile, tile_base, N, capacity, r, &kept_e);
      route_expert[r] = kept_e;
      if (over)
        for (long long q = (r / k) * k; q < r; ++q) {
          int kq = -1;
          nprev += phase_one_overflow(topk_idx, rank_in_tile, tile_base, N, capacity, q, &kq) ? 1 : 0;
        }
    }
    int total = 0;
    const int pos = n + block_scan_1024(over ? 1 : 0, wbuf, &total);
    if (over) {
      e_r[pos] = (int)r;
      e_hold[pos] = -1;
      e_ptr[pos] = 0;
      e_first[pos] = pos - nprev;
    }
    n += total;
  }
  __syncthreads();
  const int NR = N + 2;                  // rows of the exchanged counts
  const int P = kRerouteThreads / NR;    // threads per row when reading them
  const int seg = (G + P - 1) / P;       // CTAs per thread
  const int ebits = N > 1 ? 32 - __clz(N - 1) : 0;
  bool settled = false;
  int accepted = 0, round = 0;
  for (; round < max_rounds; ++round) {
    int32_t* xb = sc.lcount + (size_t)(round & 1) * xints;
    uint16_t* x_cnt = reinterpret_cast<uint16_t*>(xb);   // [N + 2][gs]
    int32_t* x_off = xb + (size_t)(N + 2) * gs / 2;      // [G][N]
    int32_t* srt = sc.lrank + (size_t)(round & 1) * R;
    // (a) proposals of the unplaced routes
    for (int j = tid; j < n; j += blockDim.x) {
      const int h = e_hold[j];
      if (h != -1) {
        e_cand[j] = h;
        continue;
      }
      const int r = e_r[j];
      const int t = r / k;
      const int f = e_first[j];   // the token's earlier overflowing slots: f .. j-1
      int p = e_ptr[j];
      int chosen = walk_list(pcache + (size_t)(t - t0) * Lc, Lc, sc.prefs + (size_t)t * L, Leff, p, r,
                             thresh, e_hold, f, j);
      e_ptr[j] = p;
      if (chosen < 0 && !lists_complete) {   // the cached list is used up: scan every expert
        uint32_t own[kMaxN / 32];
        for (int x = 0; x < kMaxN / 32; ++x) own[x] = 0u;
        for (int q = 0; q < k; ++q) {
          const int e1 = topk_idx[(long long)t * k + q];
          if (e1 >= 0 && e1 < N) own[e1 >> 5] |= 1u << (e1 & 31);
        }
        for (int q = f; q < j; ++q) {
          const int hq = e_hold[q];
          if (hq >= 0) own[hq >> 5] |= 1u << (hq & 31);
        }
        unsigned long long best = 0ull;
        for (int e = 0; e < N; ++e) {
          if (((own[e >> 5] >> (e & 31)) & 1u) || !(r < thresh[e])) continue;
          const unsigned long long key = reroute_key(logits[(size_t)t * N + e], e);
          best = key > best ? key : best;
        }
        if (best) chosen = key_expert(best);
      }
      e_cand[j] = chosen >= 0 ? chosen : -2;
    }
    for (int e = tid; e < N; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    // (b) ranks among this CTA's candidates, chunk by chunk in list order
    int dead = 0;
    for (int c0 = 0; c0 < n; c0 += kRerouteThreads) {
      const int j = c0 + tid;
      int c = -1;
      if (j < n) {
        c = e_cand[j];
        const int f = e_first[j];
#pragma unroll
        for (int d = 1; d < 16; ++d)   // the token's earlier slots: at most 15
          if (j - d >= f && e_cand[j - d] == c) c = -1;
      }
      dead += __syncthreads_count(j < n && e_cand[j] == -2);
      for (int x = tid; x < 32 * (kMaxN + 1); x += blockDim.x) (&tab[0][0])[x] = 0;
      __syncthreads();
      const unsigned peers = lanes_with_expert(c, ebits);
      const int wrank = __popc(peers & ((1u << lane) - 1u));
      if (c >= 0 && wrank == 0) tab[w][c] = __popc(peers);
      __syncthreads();
      for (int e = w; e < N; e += 32) {   // warp w: expert e's counts over the 32 warps
        const int v = tab[lane][e];
        const int carry = cnt[e];
        int incl = v;
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        tab[lane][e] = carry + incl - v;
        if (lane == 31) cnt[e] = carry + incl;
      }
      __syncthreads();
      if (j < n) e_rank[j] = c >= 0 ? tab[w][c] + wrank : -1;
      __syncthreads();
    }
    {
      int tot_c = 0;
      const int ex = block_scan_1024(tid < N ? cnt[tid] : 0, wbuf, &tot_c);
      if (tid < N) {
        off[tid] = ex;
        x_cnt[(size_t)tid * gs + X] = (uint16_t)cnt[tid];
        x_off[(size_t)X * N + tid] = ex;
      }
      if (tid == 0) {
        x_cnt[(size_t)N * gs + X] = (uint16_t)dead;
        x_cnt[(size_t)(N + 1) * gs + X] = (uint16_t)n;
      }
    }
    __syncthreads();
    for (int j = tid; j < n; j += blockDim.x)
      if (e_rank[j] >= 0) srt[r0 + off[e_cand[j]] + e_rank[j]] = e_r[j];
    if (!grid_barrier(sc.gsync, (uint32_t)G * (uint32_t)(round + 1), &s_ok, barrier_ns)) break;
    // (c) every CTA's counts
    {
      const int pieces = (N + 2) * gs / 8;   // 16-byte pieces
      for (int c = tid; c < pieces; c += blockDim.x) cp_async_16(stage + 8 * c, x_cnt + 8 * c);
    }
    cp_async_wait_all();
    __syncthreads();
    // per row: P threads sum runs of seg CTAs; then this CTA's prefix and
    // where an expert's room runs out
    if (tid < P * NR) {
      const int e = tid / P, p = tid % P;
      const uint16_t* row = stage + (size_t)e * gs;
      int v = 0;
      for (int x = p * seg; x < min(G, p * seg + seg); ++x) v += row[x];
      part[tid] = v;
    }
    __syncthreads();
    for (int e = tid; e < NR; e += blockDim.x) {
      int run = 0;
      for (int p = 0; p < P; ++p) {
        const int v = part[e * P + p];
        part[e * P + p] = run;
        run += v;
      }
      tot[e] = run;
      if (e < N) cross_x[e] = -1;
    }
    __syncthreads();
    if (tid < P * NR) {
      const int e = tid / P, p = tid % P;
      const uint16_t* row = stage + (size_t)e * gs;
      const int rm = e < N ? room[e] : 0;
      int cum = part[tid];
      for (int x = p * seg; x < min(G, p * seg + seg); ++x) {
        const int c = row[x];
        if (x == X) pre[e] = cum;
        if (e < N && rm > 0 && cum < rm && cum + c >= rm) {
          cross_x[e] = x;
          cross_q[e] = rm - 1 - cum;
        }
        cum += c;
      }
    }
    __syncthreads();
    // the route id of each full expert's last accepted candidate
    for (int e = tid; e < N; e += blockDim.x) {
      const int x = cross_x[e];
      int wr = -1;
      if (x >= 0) wr = __ldcg(&srt[(long long)x * S + __ldcg(&x_off[(size_t)x * N + e]) + cross_q[e]]);
      worst[e] = wr;
      thresh[e] = tot[e] < room[e] ? 0x7FFFFFFF : wr;
    }
    for (int j = tid; j < n; j += blockDim.x) {
      const int c = e_cand[j], rk = e_rank[j];
      e_hold[j] = (rk >= 0 && pre[c] + rk < room[c]) ? c : (c == -2 ? -2 : -1);
    }
    accepted = block_sum_1024(tid < N ? min(tot[tid], room[tid]) : 0, wbuf);
    settled = tot[N + 1] - tot[N] - accepted == 0;
    if (settled) break;
  }
  if (!s_ok) {
    if (tid == 0) {
      atomicExch(sc.flag, 1);
      atomicOr(status, kDevNoteRerouteFallback);
    }
    return;
  }
  // results: the list of overflowing routes (for the check), the targets, counts
  for (int j = tid; j < n; j += blockDim.x) {
    sc.list[pre[N + 1] + j] = e_r[j];
    route_expert[e_r[j]] = e_hold[j] >= 0 ? e_hold[j] : -1;
  }
  if (X == 0) {
    for (int e = tid; e < N; e += blockDim.x) {
      sc.acc[e] = min(tot[e], room[e]);
      sc.worst[e] = worst[e];
    }
    if (tid == 0) {
      *num_rerouted = accepted;
      *num_dropped = tot[N + 1] - accepted;
      *sc.count = tot[N + 1];
      if (!settled) atomicExch(sc.flag, 1);
    }
  }
}

// ---------------------------------------------------------------- check
// One warp per overflowing route: its target is usable, and every usable
// expert it ranks higher is full with routes of higher priority.
__global__ void __launch_bounds__(256) reroute_verify_kernel(
    const int32_t* __restrict__ topk_idx, const float* __restrict__ logits, int N, int k, int capacity,
    const int32_t* __restrict__ kept_count, RerouteScratch sc, const int32_t* __restrict__ route_expert) {
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (i >= *sc.count || *sc.flag) return;
  const int r = sc.list[i];
  const int t = r / k;
  const int target = route_expert[r];
  uint32_t used = 0;   // bit s: expert lane + 32 s is the token's own or an earlier slot's target
  for (int q = 0; q < k; ++q) {
    const int e1 = topk_idx[(long long)t * k + q];
    if (e1 >= 0 && e1 < N && (e1 & 31) == lane) used |= 1u << (e1 >> 5);
    if ((long long)t * k + q < r) {
      const int e2 = route_expert[(long long)t * k + q];
      if (e2 >= 0 && e2 < N && (e2 & 31) == lane) used |= 1u << (e2 >> 5);
    }
  }
  bool bad = false;
  if (target >= 0 && (target & 31) == lane && ((used >> (target >> 5)) & 1u)) bad = true;
  if (target >= N) bad = true;
  const unsigned long long tkey =
      target >= 0 && target < N ? reroute_key(logits[(size_t)t * N + target], target) : 0ull;
  for (int e = lane, s = 0; e < N; e += 32, ++s) {
    if ((used >> s) & 1u) continue;
    if (reroute_key(logits[(size_t)t * N + e], e) <= tkey) continue;
    const int room = capacity - kept_count[e];
    if (!(sc.acc[e] == room && sc.worst[e] < r)) bad = true;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicExch(sc.flag, 1);
}

// ---------------------------------------------------------------- sequential rule
// One CTA.  Runs only when the flag is set.  Routes are scanned in batches
// of 1024; the overflowing routes of a batch are compacted in order, then
// resolved 32 at a time, one warp each: every warp proposes its route's best
// expert given the room left, and warp 0 commits the longest prefix of
// proposals that the sequential rule would also make (no earlier unresolved
// slot of the same token, and fewer earlier proposals for the same expert
// than its room).  The first unresolved route always qualifies, so each round
// commits at least one route and a group ends within 32 rounds.
__global__ void __launch_bounds__(kRerouteThreads) reroute_seq_kernel(
    const int32_t* __restrict__ topk_idx, const float* __restrict__ logits, int T, int N, int k,
    int capacity, const int32_t* __restrict__ rank_in_tile, const int32_t* __restrict__ tile_base,
    const int32_t* __restrict__ kept_count, const int32_t* __restrict__ flag,
    int32_t* __restrict__ route_expert, int32_t* __restrict__ num_dropped,
    int32_t* __restrict__ num_rerouted) {
  if (*flag == 0) return;
  __shared__ int room[kMaxN];
  __shared__ int list[kRerouteThreads];
  __shared__ int wsum[32];
  __shared__ int tent[32];
  __shared__ int done[32];
  __shared__ int s_total, s_all_done, s_rer, s_drop;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const long long R = (long long)T * k;
  for (int e = tid; e < N; e += blockDim.x) room[e] = capacity - kept_count[e];
  if (tid == 0) {
    s_rer = 0;
    s_drop = 0;
  }
  __syncthreads();
  for (long long base = 0; base < R; base += kRerouteThreads) {
    const long long r = base + tid;
    bool over = false;
    if (r < R) {
      int kept_e = -1;
      over = phase_one_overflow(topk_idx, rank_in_tile, tile_base, N, capacity, r, &kept_e);
      route_expert[r] = kept_e;
    }
    const unsigned om = __ballot_sync(0xffffffffu, over);
    if (lane == 0) wsum[w] = __popc(om);
    __syncthreads();
    if (w == 0) {
      const int c = wsum[lane];
      int incl = c;
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      wsum[lane] = incl - c;
      if (lane == 31) s_total = incl;
    }
    __syncthreads();
    if (over) list[wsum[w] + __popc(om & ((1u << lane) - 1u))] = tid;
    __syncthreads();
    const int total = s_total;
    for (int c0 = 0; c0 < total; c0 += 32) {
      const int n = min(32, total - c0);
      if (tid < 32) done[tid] = tid < n ? 0 : 1;
      // this warp's route: token t, slot j, and the experts the token uses
      // among the experts lane, lane+32, ... (bit s = expert lane + 32 s)
      long long rr = 0;
      int t = 0;
      uint32_t used = 0;
      if (w < n) {
        rr = base + list[c0 + w];
        t = (int)(rr / k);
        for (int q = 0; q < k; ++q) {
          const long long rq = (long long)t * k + q;
          const int e1 = topk_idx[rq];
          if (e1 >= 0 && e1 < N && (e1 & 31) == lane) used |= 1u << (e1 >> 5);
        }
      }
      __syncthreads();
      for (int round = 0; round <= 32; ++round) {
        if (w < n && !done[w]) {
          const int j = (int)(rr - (long long)t * k);
          uint32_t excl = used;
          for (int q = 0; q < j; ++q) {   // targets of the token's earlier slots
            const int e2 = route_expert[(long long)t * k + q];
            if (e2 >= 0 && e2 < N && (e2 & 31) == lane) excl |= 1u << (e2 >> 5);
          }
          unsigned long long best = 0ull;
          for (int e = lane, sl = 0; e < N; e += 32, ++sl) {
            if (((excl >> sl) & 1u) || room[e] <= 0) continue;
            const unsigned long long key = reroute_key(logits[(size_t)t * N + e], e);
            best = key > best ? key : best;
          }
          for (int off = 16; off > 0; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
            best = o > best ? o : best;
          }
          if (lane == 0) tent[w] = best ? key_expert(best) : -1;
        }
        __syncthreads();
        if (w == 0) {
          const bool unres = lane < n && !done[lane];
          const int te = unres ? tent[lane] : -2;
          const long long myr = unres ? base + list[c0 + lane] : -1;
          const int tok = unres ? (int)(myr / k) : -1 - lane;
          const unsigned unres_m = __ballot_sync(0xffffffffu, unres);
          const unsigned lt = (1u << lane) - 1u;
          const bool clash = (__match_any_sync(0xffffffffu, tok) & unres_m & lt) != 0u;
          const int occ = __popc(__match_any_sync(0xffffffffu, te) & unres_m & lt);
          const bool valid = unres && !clash && (te < 0 || occ < room[te]);
          const unsigned bad = __ballot_sync(0xffffffffu, unres && !valid);
          const unsigned below = bad ? ((1u << (__ffs(bad) - 1)) - 1u) : 0xffffffffu;
          const bool commit = unres && ((below >> lane) & 1u);
          if (commit) {
            if (te >= 0) route_expert[myr] = te;
            done[lane] = 1;
          }
          const unsigned grp = __match_any_sync(0xffffffffu, commit ? te : -3 - lane);
          if (commit && te >= 0 && (grp & lt) == 0u) room[te] -= __popc(grp);
          const unsigned cr = __ballot_sync(0xffffffffu, commit && te >= 0);
          const unsigned cd = __ballot_sync(0xffffffffu, commit && te < 0);
          const unsigned left = __ballot_sync(0xffffffffu, unres && !commit);
          if (lane == 0) {
            s_rer += __popc(cr);
            s_drop += __popc(cd);
            s_all_done = left == 0u;
          }
        }
        __syncthreads();
        if (s_all_done) break;
      }
      __syncthreads();
    }
    __syncthreads();
  }
  if (tid == 0) {
    *num_dropped = s_drop;
    *num_rerouted = s_rer;
  }
}

// Grid or single-CTA rounds: forced by the caller's path flags; otherwise
// the grid from kRerouteGridMinRoutes routes on.
constexpr long long kRerouteGridMinRoutes = 16384;

bool use_grid_rounds(long long R, const PathOpts& o) {
  if (o.flags & kPathRerouteGrid) return true;
  if (o.flags & kPathRerouteOneCta) return false;
  return R >= kRerouteGridMinRoutes;
}

// Shared copy of the preference lists of a CTA's tokens: at most this many bytes.
constexpr int kListCacheBytes = 24576;

// Entries of each token's list kept in shared memory (a multiple of 16).
int list_cache_len(int tokens) {
  const int lc = tokens > 0 ? kListCacheBytes / tokens / 16 * 16 : 0;
  return lc < kRerouteListLen ? lc : kRerouteListLen;
}

// Dynamic shared memory of the grid-wide rounds: six ints per listed route,
// the 16-bit counts of every CTA, the lists' shared copy.
int grid_rounds_smem(int chunks, int G, int N, int cache_bytes) {
  return chunks * kRerouteThreads * 6 * (int)sizeof(int) +
         (N + 2) * ((G + 7) / 8 * 8) * (int)sizeof(uint16_t) + cache_bytes;
}

// Resident 1024-thread CTAs of the grid-wide rounds (one per SM at most) with
// kGridMaxChunks chunks of shared state; -1 if the kernel cannot run.
int grid_rounds_ctas() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cache[dev] != 0) return cache[dev];
  int sms0 = 0;
  cudaDeviceGetAttribute(&sms0, cudaDevAttrMultiProcessorCount, dev);
  const int smem = grid_rounds_smem(kGridMaxChunks, sms0, kMaxN, kListCacheBytes);
  int sms = 0, per = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaFuncSetAttribute(reroute_da_grid_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, reroute_da_grid_kernel, kRerouteThreads, smem) !=
          cudaSuccess) {
    cudaGetLastError();
    per = 0;
  }
  const int g = per > 0 ? sms : -1;
  if (dev >= 0 && dev < 64) cache[dev] = g;
  return g;
}

}  // namespace

void launch_reroute(const int32_t* topk_idx, const float* logits, int T, int N, int k, int capacity,
                    const int32_t* rank_in_tile, const int32_t* tile_base, const int32_t* kept_count,
                    const RerouteScratch& sc, int32_t* route_expert, int32_t* num_dropped,
                    int32_t* num_rerouted, int* status, const PathOpts& o, cudaStream_t s) {
  const long long R = (long long)T * k;
  if (o.flags & kPathRerouteSequential) {
    cudaMemsetAsync(sc.flag, 0xFF, sizeof(int32_t), s);
  } else {
    const unsigned pref_blocks = (unsigned)((T + 7) / 8);
    auto prefs = N <= 32 ? reroute_prefs_kernel<1>
               : N <= 64 ? reroute_prefs_kernel<2>
               : N <= 128 ? reroute_prefs_kernel<4> : reroute_prefs_kernel<8>;
    prefs<<<pref_blocks, 256, 0, s>>>(topk_idx, logits, T, N, k, capacity, rank_in_tile, tile_base,
                                      kRerouteListLen, sc.prefs, sc.gsync, sc.flag);
    const int max_rounds = 4 * N + 16;
    // grid-wide rounds: CTAs own whole tokens, chunks of per = k * floor(1024 / k) routes
    int gmax = use_grid_rounds(R, o) ? grid_rounds_ctas() : -1;
    if (gmax > 0 && o.grid_ctas > 0 && o.grid_ctas < gmax) gmax = o.grid_ctas;   // more routes per CTA
    const long long per = (long long)(kRerouteThreads / k) * k;
    const long long nchunks = (R + per - 1) / per;
    const int chunks = gmax > 0 ? (int)((nchunks + gmax - 1) / gmax) : 0;
    if (gmax > 0 && chunks <= kGridMaxChunks) {
      const int S = (int)(chunks * per);
      const int ctas = (int)((R + S - 1) / S);
      const int Lc = list_cache_len(S / k);
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)ctas, 1, 1);
      cfg.blockDim = dim3(kRerouteThreads, 1, 1);
      cfg.dynamicSmemBytes = (size_t)grid_rounds_smem(chunks, ctas, N, (S / k) * Lc);
      cfg.stream = s;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeCooperative;
      attr[0].val.cooperative = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaLaunchKernelEx(&cfg, reroute_da_grid_kernel, topk_idx, logits, T, N, k, capacity,
                             rank_in_tile, tile_base, kept_count, sc, kRerouteListLen, Lc, max_rounds,
                             S, chunks, route_expert, num_dropped, num_rerouted,
                             o.wait_ns ? (unsigned long long)o.wait_ns : kBarrierLimitNs, status) != cudaSuccess) {
        cudaGetLastError();   // not launched: the sequential kernel decides
        cudaMemsetAsync(sc.flag, 0xFF, sizeof(int32_t), s);
      }
    } else {
      reroute_da_kernel<<<1, kRerouteThreads, 0, s>>>(topk_idx, logits, T, N, k, capacity, rank_in_tile,
                                                      tile_base, kept_count, sc, kRerouteListLen,
                                                      max_rounds, route_expert, num_dropped,
                                                      num_rerouted);
    }
    const unsigned ver_blocks = (unsigned)((R + 7) / 8);
    reroute_verify_kernel<<<ver_blocks, 256, 0, s>>>(topk_idx, logits, N, k, capacity, kept_count, sc,
                                                     route_expert);
  }
  reroute_seq_kernel<<<1, kRerouteThreads, 0, s>>>(topk_idx, logits, T, N, k, capacity, rank_in_tile,
                                                   tile_base, kept_count, sc.flag, route_expert,
                                                   num_dropped, num_rerouted);
}

}  // namespace moe
