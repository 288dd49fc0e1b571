// Router: fp32 logits in the fixed chunked order, then top-k and renormalised
// gates ("Mixture-of-Experts Routing at Inference Time", section "How sparse
// routing works": one projection to N logits, softmax, top-k, renormalise).
//
// The logit of (token t, expert e) is, for every batch size,
//   total = +0;  for each 256-element chunk c of H (ascending):
//     part = +0;  for i in c (ascending): part = fma(h[t,i], W_g[i,e], part)
//     total = total + part
//   total = total + bias[e]
// ("Why temperature=0 Still Gives Different Answers: Batch Invariance",
// Tier 2: a reduction cut into constant 256-element pieces added in one
// order).  bf16 x bf16 products are exact in fp32, so the fma rounds exactly
// like the separate add.  Chunks are spread over the warps of a CTA and their partial sums are
// combined in ascending chunk order through shared memory; no split crosses a
// CTA and nothing depends on T.
#include <cuda_bf16.h>
#include <cstdint>

#include "kernels.h"

namespace moe {
namespace {

constexpr int kRouterWarps = 8;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// CTA tile: TT = 4*G tokens x NE = 2*P experts.  Lane l of a warp owns the
// expert pair p = l % P and the token quad g = l / P (P*G = 32).  Warp w sums
// chunks w, w+8, ...; partial sums go to part[chunk][token][expert].
template <bool kEvenN>
__global__ void __launch_bounds__(256) router_logits_kernel(const uint16_t* __restrict__ h,
                                                            const uint16_t* __restrict__ wg,
                                                            const float* __restrict__ bias,
                                                            float* __restrict__ logits, int T, int H,
                                                            int N, int P, int G) {
  extern __shared__ float part[];
  const int NE = 2 * P, TT = 4 * G;
  const int t0 = blockIdx.x * TT, e0 = blockIdx.y * NE;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p = lane % P, g = lane / P;
  const int chunks = (H + kRouterChunk - 1) / kRouterChunk;
  const int ea = e0 + 2 * p, eb = ea + 1;
  const bool va = ea < N, vb = eb < N;
  int tok[4];
  bool vt[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    tok[q] = t0 + 4 * g + q;
    vt[q] = tok[q] < T;
  }
  for (int c = warp; c < chunks; c += kRouterWarps) {
    float acc[4][2];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q][0] = acc[q][1] = 0.0f;
    const int i0 = c * kRouterChunk, i1 = min(H, i0 + kRouterChunk);
    for (int i = i0; i < i1; i += 8) {
      uint4 hv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        hv[q] = vt[q] ? __ldg(reinterpret_cast<const uint4*>(h + (size_t)tok[q] * H + i))
                      : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int ii = 0; ii < 8; ++ii) {
        float wa = 0.0f, wb = 0.0f;
        const size_t off = (size_t)(i + ii) * N + ea;
        if (kEvenN) {
          if (va) {
            uint32_t w2 = __ldg(reinterpret_cast<const unsigned int*>(wg + off));
            wa = bf16_lo(w2);
            wb = bf16_hi(w2);
          }
        } else {
          if (va) wa = __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(wg + off)) << 16);
          if (vb) wb = __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(wg + off + 1)) << 16);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t word = (ii < 2) ? hv[q].x : (ii < 4) ? hv[q].y : (ii < 6) ? hv[q].z : hv[q].w;
          const float hx = (ii & 1) ? bf16_hi(word) : bf16_lo(word);
          acc[q][0] = fmaf(hx, wa, acc[q][0]);
          acc[q][1] = fmaf(hx, wb, acc[q][1]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float* dst = part + ((size_t)c * TT + 4 * g + q) * NE + 2 * p;
      dst[0] = acc[q][0];
      dst[1] = acc[q][1];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < TT * NE; idx += blockDim.x) {
    const int tl = idx / NE, el = idx % NE;
    const int t = t0 + tl, e = e0 + el;
    if (t < T && e < N) {
      float total = 0.0f;
      for (int c = 0; c < chunks; ++c) total = total + part[((size_t)c * TT + tl) * NE + el];
      if (bias) total = total + bias[e];
      logits[(size_t)t * N + e] = total;
    }
  }
}

// Ranking: a number beats NaN; larger beats smaller; equal -> lower index.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  const bool na = isnan(va), nb = isnan(vb);
  if (na != nb) return nb;
  if (!na && va != vb) return va > vb;
  return ia < ib;
}

// One warp per token: k rounds of a warp-shuffle tournament over the N
// logits, slots sorted by expert index, gates = softmax over the selected.
__global__ void __launch_bounds__(256) topk_gates_kernel(const float* __restrict__ logits,
                                                         int32_t* __restrict__ topk_idx,
                                                         float* __restrict__ gates, int T, int N,
                                                         int k) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  float v[8];
  uint32_t used = 0;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int e = lane + 32 * s;
    if (e < N) {
      v[s] = logits[(size_t)t * N + e];
    } else {
      v[s] = 0.0f;
      used |= 1u << s;
    }
  }
  int sel[16];
  float selv[16];
  for (int j = 0; j < k; ++j) {
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
    sel[j] = bi;
    selv[j] = bv;
    if ((bi & 31) == lane) used |= 1u << (bi >> 5);
  }
  // slots in ascending expert index (insertion sort, same in every lane)
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
    topk_idx[(size_t)t * k + j] = sel[j];
    gates[(size_t)t * k + j] = ex[j] / S;
  }
}

}  // namespace

void launch_router_logits(const uint16_t* h, const uint16_t* w_gate, const float* bias, float* logits,
                          int T, int H, int N, cudaStream_t s) {
  // NE experts per CTA (power of two, 8..64), P = NE/2 pairs, G = 32/P token quads.
  int NE = 8;
  while (NE < N && NE < 64) NE *= 2;
  const int P = NE / 2, G = 32 / P, TT = 4 * G;
  const int chunks = (H + kRouterChunk - 1) / kRouterChunk;
  const size_t smem = (size_t)chunks * TT * NE * sizeof(float);
  dim3 grid((T + TT - 1) / TT, (N + NE - 1) / NE);
  if (N % 2 == 0) {
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(router_logits_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    router_logits_kernel<true><<<grid, 256, smem, s>>>(h, w_gate, bias, logits, T, H, N, P, G);
  } else {
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(router_logits_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    router_logits_kernel<false><<<grid, 256, smem, s>>>(h, w_gate, bias, logits, T, H, N, P, G);
  }
}

void launch_topk_gates(const float* logits, int32_t* topk_idx, float* gates, int T, int N, int k,
                       cudaStream_t s) {
  const int warps = 8;
  topk_gates_kernel<<<(T + warps - 1) / warps, warps * 32, 0, s>>>(logits, topk_idx, gates, T, N, k);
}

}  // namespace moe
