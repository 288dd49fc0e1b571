// Routing diagnostics: the routing_stats probe and the router margin.
//
// routing_stats ("Mixture-of-Experts Routing at Inference Time", section "The
// hard part: token dropping is a silent correctness bug"): per-expert load as
// a count of the routed expert ids, a probe capacity of floor(mean load x
// capacity factor), the overflow summed over experts, the ratio max / mean
// and the dropped fraction.  Counts are integers (shared-memory atomics give
// the same totals in any order); the three fp64 quantities are single IEEE
// operations on those integers, so every run gives the same bits.
//
// The router margin ("Mixture-of-experts routing and LLM repeatability"): the
// gap between a token's k-th and (k+1)-th logits under the router's ranking
// (larger first, equal by lower index, NaN last), as the fp64 difference of
// the two fp32 values (+inf when k = N).
#include <cstdint>

#include "kernels.h"

namespace moe {
namespace {

constexpr int kMaxN = 256;

__global__ void __launch_bounds__(1024) routing_stats_kernel(const int32_t* __restrict__ topk_idx,
                                                             long long R, int N, double cf,
                                                             int32_t* __restrict__ load_out,
                                                             RoutingStats* __restrict__ stats) {
  __shared__ int hist[kMaxN];
  for (int e = threadIdx.x; e < N; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  for (long long r = threadIdx.x; r < R; r += blockDim.x) {
    const int e = topk_idx[r];
    if (e >= 0 && e < N) atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x) load_out[e] = hist[e];
  if (threadIdx.x == 0) {
    long long total = 0;
    int mx = hist[0], mn = hist[0];
    for (int e = 0; e < N; ++e) {
      total += hist[e];
      mx = max(mx, hist[e]);
      mn = min(mn, hist[e]);
    }
    RoutingStats st{};
    if (total > 0) {
      const double mean = __ddiv_rn((double)total, (double)N);
      const int cap = (int)floor(__dmul_rn(mean, cf));
      long long drops = 0;
      for (int e = 0; e < N; ++e) drops += max(0, hist[e] - cap);
      st.max_expert_load = mx;
      st.min_expert_load = mn;
      st.capacity = cap;
      st.dropped_tokens = (int32_t)drops;
      st.total_routes = (int32_t)total;
      st.imbalance_ratio = __ddiv_rn((double)mx, mean);
      st.drop_fraction = __ddiv_rn((double)drops, (double)total);
    }
    *stats = st;
  }
}

__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  const bool na = isnan(va), nb = isnan(vb);
  if (na != nb) return nb;
  if (!na && va != vb) return va > vb;
  return ia < ib;
}

// One warp per token: k + 1 rounds of a warp tournament over the logits.
__global__ void __launch_bounds__(256) router_margin_kernel(const float* __restrict__ logits, int T,
                                                            int N, int k, double* __restrict__ margin) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  if (k >= N) {
    if (lane == 0) margin[t] = __longlong_as_double(0x7FF0000000000000ll);  // +inf
    return;
  }
  float v[8];
  uint32_t used = 0;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int e = lane + 32 * s;
    v[s] = e < N ? logits[(size_t)t * N + e] : 0.0f;
    if (e >= N) used |= 1u << s;
  }
  float kth = 0.0f, next = 0.0f;
  for (int j = 0; j <= k; ++j) {
    float bv = 0.0f;
    int bi = -1;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      if (!((used >> s) & 1u) && (bi < 0 || ranks_before(v[s], lane + 32 * s, bv, bi))) {
        bv = v[s];
        bi = lane + 32 * s;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (oi >= 0 && (bi < 0 || ranks_before(ov, oi, bv, bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) used |= 1u << (bi >> 5);
    if (j == k - 1) kth = bv;
    if (j == k) next = bv;
  }
  if (lane == 0) margin[t] = __dsub_rn((double)kth, (double)next);
}

}  // namespace

void launch_routing_stats(const int32_t* topk_idx, long long R, int N, double capacity_factor,
                          int32_t* load_out, RoutingStats* stats, cudaStream_t s) {
  routing_stats_kernel<<<1, 1024, 0, s>>>(topk_idx, R, N, capacity_factor, load_out, stats);
}

void launch_router_margin(const float* logits, int T, int N, int k, double* margin, cudaStream_t s) {
  router_margin_kernel<<<(T + 7) / 8, 256, 0, s>>>(logits, T, N, k, margin);
}

}  // namespace moe
