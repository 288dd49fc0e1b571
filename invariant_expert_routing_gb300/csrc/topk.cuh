// Top-k selection and renormalised gates of one token, shared by every
// router path (the chunked CUDA-core router, the certified tensor-core
// router and the one-launch decode front), so that all give the same bits
// ("Mixture-of-Experts routing": softmax, top-k, gates renormalised over the
// selected experts; ties to the lower expert index).
#pragma once
#include <cstdint>
#include <cmath>

namespace moe {
namespace sel {

// Ranking: a number beats NaN; larger beats smaller; equal -> lower index.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  const bool na = isnan(va), nb = isnan(vb);
  if (na != nb) return nb;
  if (!na && va != vb) return va > vb;
  return ia < ib;
}

// a beats b: a holds an entry (key >= 0) and b none, or both do and a ranks
// first.  Keys are expert indices or positions in an ascending expert list.
__device__ __forceinline__ bool beats(float va, int ka, float vb, int kb) {
  return ka >= 0 && (kb < 0 || ranks_before(va, ka, vb, kb));
}

// Bitonic sort of one (value, key) entry per lane across the warp, best
// first under ranks_before: afterwards lane p holds the p-th best entry and
// lanes without an entry (key -1) come last.  15 compare-exchange steps,
// each one shuffle pair and one comparison.
__device__ __forceinline__ void warp_sort_best_first(float& v, int& key, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, stride);
      const int ok = __shfl_xor_sync(0xffffffffu, key, stride);
      // the lower lane of a pair keeps the better entry in blocks sorted
      // best first ((lane & size) == 0), the worse one in the others
      const bool keep_better = ((lane & stride) == 0) == ((lane & size) == 0);
      const bool take = keep_better ? beats(ov, ok, v, key) : beats(v, key, ov, ok);
      if (take) {
        v = ov;
        key = ok;
      }
    }
  }
}

// Lane-parallel form of write_slots_and_gates: the lanes set in `selected`
// (at most 32) hold the selected experts in ascending expert order; the one
// with the s-th lowest lane writes slot s.  Same arithmetic as
// write_slots_and_gates: m = max selected logit, exp(l - m) per slot, the sum
// taken in slot order, each gate one division.
__device__ __forceinline__ void write_gates_lanes(unsigned selected, int e, float v, int lane,
                                                  int32_t* __restrict__ idx_out,
                                                  float* __restrict__ gate_out) {
  const bool mine = (selected >> lane) & 1u;
  float m = mine ? v : -INFINITY;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  const float ex = mine ? expf(v - m) : 0.0f;
  float S = 0.0f;
  for (unsigned mm = selected; mm != 0u; mm &= mm - 1u) S = S + __shfl_sync(0xffffffffu, ex, __ffs(mm) - 1);
  if (mine) {
    const int slot = __popc(selected & ((1u << lane) - 1u));
    idx_out[slot] = e;
    gate_out[slot] = ex / S;
  }
}

// Sorts the k selected (expert, logit) pairs by expert index and writes the
// renormalised gates exp(l_j - m) / sum_s exp(l_s - m), m = max selected,
// summed in slot order.  Every router path calls it, so all agree bitwise.
__device__ __forceinline__ void write_slots_and_gates(int (&sel)[16], float (&selv)[16], int k,
                                                      int32_t* __restrict__ idx_out,
                                                      float* __restrict__ gate_out, int lane) {
  for (int a = 1; a < k; ++a) {
    const int si = sel[a];
    const float sv = selv[a];
    int b = a - 1;
    while (b >= 0 && sel[b] > si) {
      sel[b + 1] = sel[b];
      selv[b + 1] = selv[b];
      --b;
    }
    sel[b + 1] = si;
    selv[b + 1] = sv;
  }
  float m = -INFINITY;
  for (int j = 0; j < k; ++j) m = fmaxf(m, selv[j]);
  float ex[16];
  float S = 0.0f;
  for (int j = 0; j < k; ++j) {
    ex[j] = expf(selv[j] - m);
    S = S + ex[j];
  }
  for (int j = lane; j < k; j += 32) {
    idx_out[j] = sel[j];
    gate_out[j] = ex[j] / S;
  }
}

// One warp: k rounds of a warp-shuffle tournament over the N logits of one
// token (lrow, global or shared memory, N <= 256) pick the k best; the slots
// then go in ascending expert order (ballots per group of 32 experts) and
// the gates are the softmax over the selected, with the arithmetic of
// write_slots_and_gates (m = max selected logit, exp(l - m) per slot, the sum
// in slot order, one division each).  No per-lane arrays are indexed at run
// time.
__device__ __forceinline__ void topk_select_warp(const float* lrow, int N, int k, int lane,
                                                 int32_t* __restrict__ idx_out,
                                                 float* __restrict__ gate_out) {
  float v[8];
  uint32_t avail = 0;   // bit s: expert lane + 32 s exists and is not taken yet
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int e = lane + 32 * s;
    v[s] = 0.0f;
    if (e < N) {
      v[s] = lrow[e];
      avail |= 1u << s;
    }
  }
  const uint32_t present = avail;
  for (int j = 0; j < k; ++j) {
    float bv = 0.0f;
    int bi = -1;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      if (((avail >> s) & 1u) && (bi < 0 || ranks_before(v[s], lane + 32 * s, bv, bi))) {
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
    if (bi >= 0 && (bi & 31) == lane) avail &= ~(1u << (bi >> 5));
  }
  const uint32_t chosen = present & ~avail;
  unsigned M[8];
  float m = -INFINITY;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    M[s] = __ballot_sync(0xffffffffu, (chosen >> s) & 1u);
    if ((chosen >> s) & 1u) m = fmaxf(m, v[s]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float ex[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) ex[s] = ((chosen >> s) & 1u) ? expf(v[s] - m) : 0.0f;
  float S = 0.0f;
#pragma unroll
  for (int s = 0; s < 8; ++s)
    for (unsigned mm = M[s]; mm != 0u; mm &= mm - 1u) S = S + __shfl_sync(0xffffffffu, ex[s], __ffs(mm) - 1);
  int base = 0;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    if ((chosen >> s) & 1u) {
      const int slot = base + __popc(M[s] & ((1u << lane) - 1u));
      idx_out[slot] = lane + 32 * s;
      gate_out[slot] = ex[s] / S;
    }
    base += __popc(M[s]);
  }
}

}  // namespace sel
}  // namespace moe
