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
// rounds run in one CTA (reroute_da_kernel); proposals walk a cached list of
// each route's best experts (reroute_prefs_kernel), with a full scan once the
// list is used up.  The outcome is then checked against a characterisation of
// the sequential rule (reroute_verify_kernel): every target is usable, and
// every usable expert a route ranks above its outcome is full with routes of
// higher priority.  An assignment that passes is the sequential one (at each
// route's turn its target had room and every better usable expert did not).
// If the check fails or the rounds do not settle, reroute_seq_kernel, a
// direct implementation of the sequential rule, recomputes the assignment.
// Every decision is on integers, so the result is the same bits either way.
#include <cstdint>
#include <cstdlib>

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
// One warp per route; for an overflowing route, its first min(L, N - k)
// experts outside its own top-k, best first.
__global__ void __launch_bounds__(256) reroute_prefs_kernel(
    const int32_t* __restrict__ topk_idx, const float* __restrict__ logits, long long R, int N, int k,
    int capacity, const int32_t* __restrict__ rank_in_tile, const int32_t* __restrict__ tile_base,
    int L, uint8_t* __restrict__ prefs) {
  const int lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= R) return;
  int kept_e = -1;
  const bool over = phase_one_overflow(topk_idx, rank_in_tile, tile_base, N, capacity, r, &kept_e);
  if (!over) return;
  const long long t = r / k;
  unsigned long long key[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int e = lane + 32 * s;
    key[s] = e < N ? reroute_key(logits[(size_t)t * N + e], e) : 0ull;
  }
  for (int q = 0; q < k; ++q) {   // the token's own experts are not candidates
    const int e = topk_idx[t * k + q];
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (e == lane + 32 * s) key[s] = 0ull;
  }
  const int n = min(L, N - k);
  for (int p = 0; p < n; ++p) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int s = 0; s < 8; ++s) best = key[s] > best ? key[s] : best;
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
      best = o > best ? o : best;
    }
    const int e = key_expert(best);
    if (lane == 0) prefs[(size_t)r * L + p] = (uint8_t)e;
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (e == lane + 32 * s) key[s] = 0ull;
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

// ---------------------------------------------------------------- deferred acceptance
// hold[i] (list position i): the expert route list[i] holds, -1 none yet,
// -2 no expert can take it any more.  cnt/worst: after each round, how many
// overflow routes each expert holds and the largest such route id (-1 none);
// an expert can still take route r if cnt < room or worst > r.
__global__ void __launch_bounds__(kRerouteThreads) reroute_da_kernel(
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
      int held[16];
      int nh = 0;
      for (int q = sc.first[i]; q < i; ++q) {   // the token's earlier overflowing slots
        const int hq = sc.hold[q];
        if (hq >= 0) held[nh++] = hq;
      }
      int chosen = -1;
      int p = sc.ptr[i];
      // walk the cached list 16 entries (one 16-byte load) at a time
      const uint4* row = reinterpret_cast<const uint4*>(sc.prefs + (size_t)r * L);
      while (p < Leff && chosen < 0) {
        const uint4 v = row[p >> 4];
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
        for (int b = p & 15; b < 16 && p < Leff; ++b, ++p) {
          const int e = (int)((wv[b >> 2] >> (8 * (b & 3))) & 0xFFu);
          bool ex = false;
          for (int x = 0; x < nh; ++x) ex |= held[x] == e;
          if (!ex && r < thresh[e]) {
            chosen = e;
            break;
          }
        }
      }
      sc.ptr[i] = p;
      if (chosen < 0 && !lists_complete) {
        // the cached list is used up: scan every expert
        uint32_t own[kMaxN / 32];
        for (int x = 0; x < kMaxN / 32; ++x) own[x] = 0u;
        for (int q = 0; q < k; ++q) {
          const int e1 = topk_idx[(long long)t * k + q];
          if (e1 >= 0 && e1 < N) own[e1 >> 5] |= 1u << (e1 & 31);
        }
        for (int x = 0; x < nh; ++x) own[held[x] >> 5] |= 1u << (held[x] & 31);
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

bool force_sequential() {
  static const bool v = [] {
    const char* s = std::getenv("MOE_REROUTE_SEQUENTIAL");
    return s && s[0] == '1';
  }();
  return v;
}

}  // namespace

void launch_reroute(const int32_t* topk_idx, const float* logits, int T, int N, int k, int capacity,
                    const int32_t* rank_in_tile, const int32_t* tile_base, const int32_t* kept_count,
                    const RerouteScratch& sc, int32_t* route_expert, int32_t* num_dropped,
                    int32_t* num_rerouted, cudaStream_t s) {
  const long long R = (long long)T * k;
  if (force_sequential()) {
    cudaMemsetAsync(sc.flag, 0xFF, sizeof(int32_t), s);
  } else {
    const unsigned pref_blocks = (unsigned)((R + 7) / 8);
    reroute_prefs_kernel<<<pref_blocks, 256, 0, s>>>(topk_idx, logits, R, N, k, capacity, rank_in_tile,
                                                     tile_base, kRerouteListLen, sc.prefs);
    const int max_rounds = 4 * N + 16;
    reroute_da_kernel<<<1, kRerouteThreads, 0, s>>>(topk_idx, logits, T, N, k, capacity, rank_in_tile,
                                                    tile_base, kept_count, sc, kRerouteListLen,
                                                    max_rounds, route_expert, num_dropped, num_rerouted);
    const unsigned ver_blocks = (unsigned)((R + 7) / 8);
    reroute_verify_kernel<<<ver_blocks, 256, 0, s>>>(topk_idx, logits, N, k, capacity, kept_count, sc,
                                                     route_expert);
  }
  reroute_seq_kernel<<<1, kRerouteThreads, 0, s>>>(topk_idx, logits, T, N, k, capacity, rank_in_tile,
                                                   tile_base, kept_count, sc.flag, route_expert,
                                                   num_dropped, num_rerouted);
}

}  // namespace moe
