// Expert-choice routing ("Mixture-of-experts routing and LLM repeatability":
// each expert takes its highest-scoring tokens of the batch; "Mixture-of-
// Experts Routing at Inference Time", section "Integration: where routing
// lives in a serving stack", the comparison of routing variants: each expert
// picks the tokens it will take, up to its capacity).
//
// Scores are the router's softmax probabilities.  For a fixed expert the
// ranking of tokens by probability is decided in fp64 on the log scale:
//   key[t,e] = (l[t,e] - m_t) - log(sum over e' ascending of exp(l[t,e'] - m_t))
// (m_t = largest non-NaN logit; NaN logits are left out of the sum and rank
// last).  l - m is exact in fp64 and the sum runs in one order, so tokens whose
// logits differ by a constant get identical keys, and the key of a token does
// not depend on the batch.  Expert e takes the C tokens with the largest keys,
// equal keys by lower token index; the probability exp(key) is its gate.
//
// Routes are r = t*N + e.  Every expert takes exactly min(C, T) tokens, so the
// padded layout is known in closed form: expert e's segment starts at
// e * P, P = min(C, T) rounded up to B, and holds its tokens in ascending t.
#include <cstdint>

#include "kernels.h"

namespace moe {
namespace {

constexpr int kEcThreads = 1024;

// Sortable form of an fp64 key: larger key -> larger integer; NaN -> 0.
__device__ __forceinline__ unsigned long long ec_sortable(double k) {
  if (isnan(k)) return 0ull;
  unsigned long long u = (unsigned long long)__double_as_longlong(k);
  if (u == 0x8000000000000000ull) u = 0ull;
  return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}

// One warp per token: keys [N][T] (sortable, transposed for the per-expert
// selection) and gates [T][N] = fp32(exp(key)).
__global__ void __launch_bounds__(256) ec_score_kernel(const float* __restrict__ logits, int T, int N,
                                                       unsigned long long* __restrict__ keys,
                                                       float* __restrict__ gates) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  float v[8];
  double m = -__longlong_as_double(0x7FF0000000000000ll);  // -inf
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int e = lane + 32 * s;
    v[s] = e < N ? logits[(size_t)t * N + e] : __int_as_float(0x7FC00000);
    if (!isnan(v[s])) m = fmax(m, (double)v[s]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmax(m, __shfl_xor_sync(0xffffffffu, m, off));
  double term[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) term[s] = isnan(v[s]) ? 0.0 : exp(__dsub_rn((double)v[s], m));
  // the sum in ascending expert order: expert e's term lives in lane e % 32
  // (a NaN logit's term is +0, which leaves the sum unchanged: the same
  // bits as leaving it out)
  double sum = 0.0;
  for (int e = 0; e < N; ++e) {
    double x = 0.0;
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (s == (e >> 5)) x = __shfl_sync(0xffffffffu, term[s], e & 31);
    sum = __dadd_rn(sum, x);
  }
  const double log_s = log(sum);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int e = lane + 32 * s;
    if (e < N) {
      const double key = isnan(v[s]) ? __longlong_as_double(0x7FF8000000000000ll)
                                     : __dsub_rn(__dsub_rn((double)v[s], m), log_s);
      keys[(size_t)e * T + t] = ec_sortable(key);
      gates[(size_t)t * N + e] = (float)exp(key);
    }
  }
}

// Block-wide exclusive scan of one int per thread (kEcThreads threads).
__device__ int ec_block_scan(int v, int* wbuf, int* total) {
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
  const int r = wbuf[w] + incl - v;
  *total = wbuf[32];
  __syncthreads();
  return r;
}

// One CTA per expert.  Radix select (8 bits per pass, most significant
// first) finds the C-th largest key K; the expert takes every token with a
// larger key and the first C - #larger tokens (ascending t) whose key equals
// K.  Then the segment is written in ascending t and padded with R = T*N.
__global__ void __launch_bounds__(kEcThreads) ec_select_kernel(
    const unsigned long long* __restrict__ keys, int T, int N, int C, int B, uint8_t* __restrict__ route_kept,
    int32_t* __restrict__ route_pos, int32_t* __restrict__ sorted_route_ids,
    int32_t* __restrict__ block_expert, int32_t* __restrict__ num_padded,
    int32_t* __restrict__ expert_counts) {
  __shared__ int hist[256];
  __shared__ int wbuf[33];
  __shared__ unsigned long long s_prefix;
  __shared__ int s_need;
  const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const unsigned long long* ke = keys + (size_t)e * T;
  const int P = (C + B - 1) / B * B;
  const int seg = e * P;
  if (tid == 0) {
    s_prefix = 0ull;
    s_need = C;
  }
  __syncthreads();
  unsigned long long mask = 0ull;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const unsigned long long prefix = s_prefix;
    for (int t = tid; t < T; t += blockDim.x) {
      const unsigned long long k = ke[t];
      if ((k & mask) == prefix) atomicAdd(&hist[(int)((k >> shift) & 255ull)], 1);
    }
    __syncthreads();
    if (tid < 32) {
      const int need = s_need;
      // lane l holds digits 255-8l .. 248-8l (high digits first)
      int c[8], lsum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = hist[255 - 8 * lane - i];
        lsum += c[i];
      }
      int incl = lsum;
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const int before = incl - lsum;   // keys with a higher digit than this lane's
      __syncwarp();
      if (before < need && need <= incl) {
        int cum = before, d = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (cum + c[i] >= need) {
            d = 255 - 8 * lane - i;
            break;
          }
          cum += c[i];
        }
        s_prefix = prefix | ((unsigned long long)d << shift);
        s_need = need - cum;
      }
    }
    mask |= 255ull << shift;
    __syncthreads();
  }
  const unsigned long long K = s_prefix;
  const int take_eq = s_need;   // how many tokens with key == K are taken
  int eq_base = 0, sel_base = 0;
  for (int t0 = 0; t0 < T; t0 += blockDim.x) {
    const int t = t0 + tid;
    const unsigned long long k = t < T ? ke[t] : 0ull;
    const bool gt = t < T && k > K;
    const bool eq = t < T && k == K;
    int eq_tot = 0;
    const int eq_rank = eq_base + ec_block_scan(eq ? 1 : 0, wbuf, &eq_tot);
    const bool sel = gt || (eq && eq_rank < take_eq);
    int sel_tot = 0;
    const int pos = sel_base + ec_block_scan(sel ? 1 : 0, wbuf, &sel_tot);
    if (t < T) {
      const size_t r = (size_t)t * N + e;
      route_kept[r] = sel ? 1 : 0;
      route_pos[r] = sel ? seg + pos : -1;
      if (sel) sorted_route_ids[seg + pos] = (int32_t)r;
    }
    eq_base += eq_tot;
    sel_base += sel_tot;
  }
  const int R = T * N;
  for (int j = C + tid; j < P; j += blockDim.x) sorted_route_ids[seg + j] = R;
  for (int b = tid; b < P / B; b += blockDim.x) block_expert[e * (P / B) + b] = e;
  if (tid == 0) {
    expert_counts[e] = C;
    if (e == 0) *num_padded = N * P;
  }
}

}  // namespace

void launch_expert_choice(const float* logits, int T, int N, int C, int B, unsigned long long* keys,
                          float* gates, uint8_t* route_kept, int32_t* route_pos, int32_t* sorted_route_ids,
                          int32_t* block_expert, int32_t* num_padded, int32_t* expert_counts,
                          cudaStream_t s) {
  ec_score_kernel<<<(T + 7) / 8, 256, 0, s>>>(logits, T, N, keys, gates);
  ec_select_kernel<<<N, kEcThreads, 0, s>>>(keys, T, N, C, B, route_kept, route_pos, sorted_route_ids,
                                            block_expert, num_padded, expert_counts);
}

}  // namespace moe
