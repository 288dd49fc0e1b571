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
// like the separate add.  Three implementations give these bits: the chunked
// CUDA-core router (router_partials_kernel + router_reduce_kernel: chunk sums
// in parallel CTAs, added in ascending chunk order per token), its decode
// form (the same chunk sums, then one CTA of the dispatch code adds them in
// the same order), and the certified tensor-core router (route_certified_kernel
// filters the candidates, cert_chunk_kernel recomputes their chunk sums in
// the same order from shared-memory tiles, cert_finalize_kernel adds them);
// the split of work never changes a logit's order and nothing depends on T.
#include <cuda_bf16.h>
#include <cstdint>

#include "kernels.h"
#include "pdl.cuh"
#include "topk.cuh"

namespace moe {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

using sel::ranks_before;
using sel::topk_select_warp;
using sel::write_slots_and_gates;

// Chunked router on the CUDA cores: two launches, for a few tokens (decode)
// and for batches when W_g is small.
//
// router_partials_kernel: one CTA per (256-element chunk c of H, LE experts,
// TB tokens).  The CTA copies the chunk's W_g rows for its experts and its
// tokens' row slices into shared memory (cp.async, one round trip); lane l of
// a warp serves expert l % LE for token group l / LE, and each thread runs
// the in-order fma chains of chunk c for TQ tokens (interleaved, so that the
// token groups of a warp read different banks), writing the chunk sums.
// router_reduce_kernel: one CTA per token adds the chunk sums in ascending
// chunk order, then the bias, and (unless only logits are wanted) selects
// the top-k with the warp tournament of topk_select_warp.
constexpr int kPartWarps = 8;
constexpr int kPartRow = kRouterChunk + 8;   // token row stride in shared memory (528 B)

__device__ __forceinline__ void cp_async_16(void* smem, const void* gmem) {
  const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}

template <bool kVec, int LE, int TQ, int EQ>
__global__ void __launch_bounds__(kPartWarps * 32) router_partials_kernel(
    const uint16_t* __restrict__ h, const uint16_t* __restrict__ wg, int T, int H, int N,
    float* __restrict__ part) {
  pdl_wait();      // earlier kernels' outputs are visible from here on
  pdl_trigger();
  constexpr int EG = LE / EQ;                // expert groups of EQ per warp row
  constexpr int G = 32 / EG;                 // token groups per warp
  constexpr int TB = kPartWarps * G * TQ;    // tokens per CTA
  extern __shared__ __align__(16) uint16_t psm[];
  uint16_t* sw = psm;                        // [256][LE] W_g rows of the chunk
  uint16_t* sx = psm + kRouterChunk * LE;    // [TB][kPartRow] token row slices
  const int chunks = (H + kRouterChunk - 1) / kRouterChunk;
  const int c = blockIdx.x, e0 = blockIdx.y * LE, t0 = blockIdx.z * TB;
  const int i0 = c * kRouterChunk, len = min(H, i0 + kRouterChunk) - i0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ne = min(LE, N - e0);
  const int nt = min(TB, T - t0);
  if (kVec) {   // N % 8 == 0, H % 8 == 0, 16-byte aligned W_g and h: 16-byte pieces
    const int per_row = ne / 8;
    for (int idx = tid; idx < len * per_row; idx += blockDim.x) {
      const int r = idx / per_row, q = idx % per_row;
      cp_async_16(sw + r * LE + 8 * q, wg + (size_t)(i0 + r) * N + e0 + 8 * q);
    }
    const int vec = len / 8;
    for (int idx = tid; idx < nt * vec; idx += blockDim.x) {
      const int q = idx / vec, v = idx % vec;
      cp_async_16(sx + q * kPartRow + 8 * v, h + (size_t)(t0 + q) * H + i0 + 8 * v);
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  } else {
    for (int idx = tid; idx < len * LE; idx += blockDim.x) {
      const int r = idx / LE, e = idx % LE;
      sw[r * LE + e] = e < ne ? wg[(size_t)(i0 + r) * N + e0 + e] : (uint16_t)0;
    }
    for (int idx = tid; idx < nt * len; idx += blockDim.x) {
      const int q = idx / len, i = idx % len;
      sx[q * kPartRow + i] = h[(size_t)(t0 + q) * H + i0 + i];
    }
  }
  __syncthreads();
  const int el = (lane % EG) * EQ, tg = lane / EG;
  if (el >= ne) return;
  const int tb = warp * G * TQ + tg;         // this thread's tokens: tb + G * q
  float p[TQ][EQ];
#pragma unroll
  for (int q = 0; q < TQ; ++q)
#pragma unroll
    for (int u = 0; u < EQ; ++u) p[q][u] = 0.0f;
  // two elements per step (chunk lengths are multiples of 128); each chain
  // takes element i, then i + 1
#pragma unroll 4
  for (int i = 0; i < len; i += 2) {
    float w0[EQ], w1[EQ];
    if (EQ == 4) {
      const uint2 a0 = *reinterpret_cast<const uint2*>(sw + i * LE + el);
      const uint2 a1 = *reinterpret_cast<const uint2*>(sw + (i + 1) * LE + el);
      w0[0] = bf16_lo(a0.x);
      w0[1 % EQ] = bf16_hi(a0.x);
      w0[2 % EQ] = bf16_lo(a0.y);
      w0[3 % EQ] = bf16_hi(a0.y);
      w1[0] = bf16_lo(a1.x);
      w1[1 % EQ] = bf16_hi(a1.x);
      w1[2 % EQ] = bf16_lo(a1.y);
      w1[3 % EQ] = bf16_hi(a1.y);
    } else {
#pragma unroll
      for (int u = 0; u < EQ; ++u) {
        w0[u] = __uint_as_float((uint32_t)sw[i * LE + el + u] << 16);
        w1[u] = __uint_as_float((uint32_t)sw[(i + 1) * LE + el + u] << 16);
      }
    }
#pragma unroll
    for (int q = 0; q < TQ; ++q) {
      const uint32_t hw = *reinterpret_cast<const uint32_t*>(sx + (tb + G * q) * kPartRow + i);
      const float h0 = bf16_lo(hw), h1 = bf16_hi(hw);
#pragma unroll
      for (int u = 0; u < EQ; ++u) {
        p[q][u] = fmaf(h0, w0[u], p[q][u]);
        p[q][u] = fmaf(h1, w1[u], p[q][u]);
      }
    }
  }
#pragma unroll
  for (int q = 0; q < TQ; ++q) {
    const int tl = tb + G * q;
    if (tl >= nt) continue;
#pragma unroll
    for (int u = 0; u < EQ; ++u)
      if (el + u < ne) part[((size_t)(t0 + tl) * chunks + c) * N + e0 + el + u] = p[q][u];
  }
}

__global__ void __launch_bounds__(256) router_reduce_kernel(const float* __restrict__ part,
                                                            const float* __restrict__ bias, int T, int N,
                                                            int chunks, int k, float* __restrict__ logits,
                                                            int32_t* __restrict__ topk_idx,
                                                            float* __restrict__ gates) {
  pdl_wait();      // earlier kernels' outputs are visible from here on
  pdl_trigger();
  // one CTA per token, one thread per expert: the chunk sums are loaded eight
  // at a time (independent loads), then added in ascending chunk order
  __shared__ float lrow[256];
  const int t = blockIdx.x, e = threadIdx.x;
  if (e < N) {
    const float* pe = part + (size_t)t * chunks * N + e;
    float total = 0.0f;
    for (int c0 = 0; c0 < chunks; c0 += 8) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = c0 + j < chunks ? pe[(size_t)(c0 + j) * N] : 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (c0 + j < chunks) total = total + v[j];
    }
    if (bias) total = total + bias[e];
    lrow[e] = total;
    if (logits) logits[(size_t)t * N + e] = total;
  }
  __syncthreads();
  if (topk_idx && threadIdx.x < 32)
    topk_select_warp(lrow, N, k, threadIdx.x, topk_idx + (size_t)t * k, gates + (size_t)t * k);
}

// ------------------------------------------------------------------------
// Tensor-core router with a certified candidate filter.
//
// The logits are also computed on the tensor cores (the grouped GEMM kernel
// in identity mode, W_g as the weights operand): l_tc.  tcgen05 does not
// publish its accumulation order, so l_tc is used only to exclude experts
// that provably cannot enter the top-k.  With S = sum_i |h_i w_ie| <=
// ||h_t|| ||w_e|| (Cauchy-Schwarz), the tensor-core result and the canonical
// fp32 result of the chunked order both lie within their error bounds of the
// exact dot product, so |l_tc - l_canonical| <= delta_t = beta ||h_t||
// max_e ||w_e|| (+ the bias roundings), beta covering (K/16 + 1) MMA steps at
// a per-step relative error of 2^-20 and the (256 + chunks + 1) fp32
// additions of the canonical order.  If L_k is the k-th largest l_tc, every
// expert with l_tc < L_k - 2 delta_t has a canonical logit strictly below the
// canonical k-th value, so only the remaining candidates get their canonical
// logits computed (in the canonical chunked order), and the
// top-k and gates are chosen from those.  The indices and gates are
// therefore bit-identical to the CUDA-core router's; only the work differs.
// Every decision depends on the token's own values alone.

// W_g prepared for the certified router in one launch: blocks below
// `tblocks` transpose 32 x 32 tiles of W_g [H, N] into wgT [N, H] (the
// candidates' rows for the recompute); the others each compute
// norm_w[e] >= ||W_g[:, e]||_2 for eight experts from W_g itself (fp32 sums
// of squares in a fixed order, scaled up to cover their rounding).
__global__ void __launch_bounds__(256) gate_prep_kernel(const uint16_t* __restrict__ wg,
                                                        uint16_t* __restrict__ wgT,
                                                        float* __restrict__ norm_w, int H, int N,
                                                        int tblocks) {
  pdl_wait();      // earlier kernels' outputs are visible from here on
  pdl_trigger();
  __shared__ uint16_t tile[32][33];
  __shared__ float part[256][9];
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
  if ((int)blockIdx.x < tblocks) {
    const int ex = (N + 31) / 32;
    const int e0 = (blockIdx.x % ex) * 32, i0 = (blockIdx.x / ex) * 32;
    for (int r = ty; r < 32; r += 8) {
      const int i = i0 + r, e = e0 + tx;
      tile[r][tx] = (i < H && e < N) ? wg[(size_t)i * N + e] : 0;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
      const int e = e0 + r, i = i0 + tx;
      if (e < N && i < H) wgT[(size_t)e * H + i] = tile[tx][r];
    }
    return;
  }
  // eight experts e0 .. e0+7 (N % 8 == 0): thread t sums rows t, t+256, ...
  // (one 16-byte load per row), then expert q adds the 256 partial sums in
  // thread order
  const int e0 = ((int)blockIdx.x - tblocks) * 8;
  float ss[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int i = tid; i < H; i += 256) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(wg + (size_t)i * N + e0));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16_lo(w[j]), b = bf16_hi(w[j]);
      ss[2 * j] = fmaf(a, a, ss[2 * j]);
      ss[2 * j + 1] = fmaf(b, b, ss[2 * j + 1]);
    }
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) part[tid][q] = ss[q];
  __syncthreads();
  if (tid < 8) {
    float t = 0.0f;
    for (int r = 0; r < 256; ++r) t += part[r][tid];
    norm_w[e0 + tid] = sqrtf(t * (1.0f + 0x1p-7f)) * (1.0f + 0x1p-7f);
  }
}

constexpr int kCertWarps = 8;
constexpr int kCertMaxH = 8192;   // rows up to 32 chunks: one chunk per lane at most
constexpr int kCertPass = 16;     // candidates whose canonical logits one pass evaluates
constexpr int kCertQ = 32;        // candidates per token handed to the tiled recompute
constexpr int kCertTT = 32;       // tokens per tile of the tiled recompute (at most 128)
constexpr int kCertWRows = 48;    // expert rows one pass of the tiled recompute stages
constexpr int kCertRow = kRouterChunk * 2 + 16;   // 528-byte shared row: 16-byte pieces conflict-free

// The filter: one warp per token computes ||h_t||, the bound and the
// candidate list.  A token with at most kCertQ candidates hands the list to
// the tiled recompute (cand, ccount); one with more (a near-tied or
// non-finite row) is finished here: its candidates' canonical logits in
// passes of kCertPass (lane = chunk, four chains at a time), then the top-k.
// Shared memory per warp: candidate list and canonical values, and the chunk
// partial sums of one pass of candidates.
struct CertSmem {
  int cidx[kCertWarps][256];
  float cval[kCertWarps][256];
  float part[kCertWarps][kCertPass * 32];
};

__global__ void __launch_bounds__(kCertWarps * 32) route_certified_kernel(
    const float* __restrict__ logits_tc, const float* __restrict__ bias, const uint16_t* __restrict__ h,
    const uint16_t* __restrict__ wgT, const float* __restrict__ norm_w, int T, int H, int N, int k,
    float beta, int32_t* __restrict__ topk_idx, float* __restrict__ gates, int32_t* __restrict__ n_cand,
    int32_t* __restrict__ cand, int32_t* __restrict__ ccount) {
  pdl_wait();      // earlier kernels' outputs are visible from here on
  pdl_trigger();
  __shared__ CertSmem sm;
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kCertWarps + wib;
  if (t >= T) return;
  const unsigned full = 0xffffffffu;
  const uint16_t* hrow = h + (size_t)t * H;
  // ||h_t||^2
  float ss = 0.0f;
  for (int i = lane * 8; i < H; i += 256) {
    const uint4 hv = __ldg(reinterpret_cast<const uint4*>(hrow + i));
    const uint32_t w[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16_lo(w[j]), b = bf16_hi(w[j]);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
  // tensor-core logits (+ bias) of the experts this lane holds, and the
  // lane's best one under the ranking
  float v[8];
  uint32_t present = 0;
  float vmax_abs = 0.0f, lane_best = 0.0f;
  int lane_best_e = -1;
  bool finite = true;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int e = lane + 32 * s;
    v[s] = 0.0f;
    if (e < N) {
      v[s] = logits_tc[(size_t)t * N + e] + (bias ? bias[e] : 0.0f);
      present |= 1u << s;
      finite = finite && isfinite(v[s]);
      vmax_abs = fmaxf(vmax_abs, fabsf(v[s]));
      if (lane_best_e < 0 || ranks_before(v[s], e, lane_best, lane_best_e)) {
        lane_best = v[s];
        lane_best_e = e;
      }
    }
  }
  float wmax = 0.0f;
  for (int e = lane; e < N; e += 32) wmax = fmaxf(wmax, norm_w[e]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    ss += __shfl_xor_sync(full, ss, off);
    wmax = fmaxf(wmax, __shfl_xor_sync(full, wmax, off));
    vmax_abs = fmaxf(vmax_abs, __shfl_xor_sync(full, vmax_abs, off));
  }
  finite = __all_sync(full, finite);
  const float hn = sqrtf(ss * (1.0f + 0x1p-7f)) * (1.0f + 0x1p-7f);
  const float delta = beta * hn * wmax * (1.0f + 0x1p-6f) + 0x1p-21f * vmax_abs;
  finite = finite && isfinite(delta);
  // V = k-th best of the 32 lane bests: at least k experts have l_tc >= V,
  // so the canonical k-th logit is >= V - delta and every expert with
  // l_tc < V - 2 delta is out.  (N >= 128 here: every lane holds experts.)
  float V = lane_best;
  {
    // the lane bests sorted best first; V is the k-th
    int vk = lane_best_e;
    sel::warp_sort_best_first(V, vk, lane);
    V = __shfl_sync(full, V, k - 1);
  }
  const float cut = V - 2.0f * delta;
  int nc = 0;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const bool is_cand = ((present >> s) & 1u) && (!finite || v[s] >= cut);
    const unsigned m = __ballot_sync(full, is_cand);
    if (is_cand) sm.cidx[wib][nc + __popc(m & ((1u << lane) - 1u))] = lane + 32 * s;
    nc += __popc(m);
  }
  __syncwarp();
  if (n_cand && lane == 0) n_cand[t] = nc;
  if (nc <= kCertQ) {
    // the usual case: the tiled kernels finish this token
    if (lane < nc) cand[(size_t)t * kCertQ + lane] = sm.cidx[wib][lane];
    if (lane == 0) ccount[t] = nc;
    return;
  }
  if (lane == 0) ccount[t] = -1;   // finished here
  // canonical logits of the candidates.  Lane (chunk c, group g): c = lane %
  // C, g = lane / C, G = 32 / C groups; it sums chunk c from +0 in ascending
  // index with fma for the pass's candidates q = g, g+G, ... (four at a time,
  // sharing the unpacked token values).  Then each candidate's chunk sums
  // are added to +0 in ascending chunk order, then the bias.
  const int C = (H + kRouterChunk - 1) / kRouterChunk;
  const int G = 32 / C;
  const int c = lane % C, g = lane / C;
  const bool active = g < G;
  const int i0 = c * kRouterChunk, len = min(H, i0 + kRouterChunk) - i0;
  float* part = sm.part[wib];
  for (int q0 = 0; q0 < nc; q0 += kCertPass) {
    const int nq = min(kCertPass, nc - q0);
    for (int qb = g; active && qb < nq; qb += 4 * G) {
      int ce[4];
      float acc[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = qb + u * G;
        ce[u] = (q < nq) ? sm.cidx[wib][q0 + q] : -1;
        acc[u] = 0.0f;
      }
      // 16 elements (two full 32-byte sectors) per step; chunk lengths are
      // multiples of 128
      for (int i = 0; i < len; i += 16) {
        const uint4 hv0 = __ldg(reinterpret_cast<const uint4*>(hrow + i0 + i));
        const uint4 hv1 = __ldg(reinterpret_cast<const uint4*>(hrow + i0 + i + 8));
        const uint32_t hw[8] = {hv0.x, hv0.y, hv0.z, hv0.w, hv1.x, hv1.y, hv1.z, hv1.w};
        float hx[16];
#pragma unroll
        for (int ii = 0; ii < 16; ++ii) hx[ii] = (ii & 1) ? bf16_hi(hw[ii >> 1]) : bf16_lo(hw[ii >> 1]);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (ce[u] < 0) continue;
          const uint4* wp = reinterpret_cast<const uint4*>(wgT + (size_t)ce[u] * H + i0 + i);
          const uint4 wv0 = __ldg(wp), wv1 = __ldg(wp + 1);
          const uint32_t ww[8] = {wv0.x, wv0.y, wv0.z, wv0.w, wv1.x, wv1.y, wv1.z, wv1.w};
#pragma unroll
          for (int ii = 0; ii < 16; ++ii) {
            const float wx = (ii & 1) ? bf16_hi(ww[ii >> 1]) : bf16_lo(ww[ii >> 1]);
            acc[u] = fmaf(hx[ii], wx, acc[u]);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (ce[u] >= 0) part[(qb + u * G) * C + c] = acc[u];
    }
    __syncwarp();
    if (lane < nq) {
      float total = 0.0f;
      for (int cc = 0; cc < C; ++cc) total = total + part[lane * C + cc];
      const int e = sm.cidx[wib][q0 + lane];
      if (bias) total = total + bias[e];
      sm.cval[wib][q0 + lane] = total;
    }
    __syncwarp();
  }
  // top-k among the candidates: k rounds of a warp tournament (the same
  // ranking; candidates past the first 32 per lane are folded in by a loop)
  int sel[16];
  float selv[16];
  uint32_t taken = 0;   // bit s: candidate lane + 32 s already selected (nc <= 256)
  for (int j = 0; j < k; ++j) {
    float bv = 0.0f;
    int bi = -1, bs = -1;
    for (int q = lane, sl = 0; q < nc; q += 32, ++sl) {
      if ((taken >> sl) & 1u) continue;
      const int e = sm.cidx[wib][q];
      const float cv = sm.cval[wib][q];
      if (bi < 0 || ranks_before(cv, e, bv, bi)) {
        bv = cv;
        bi = e;
        bs = sl;
      }
    }
    int bq = bs >= 0 ? lane + 32 * bs : -1;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(full, bv, off);
      const int oi = __shfl_xor_sync(full, bi, off);
      const int oq = __shfl_xor_sync(full, bq, off);
      if (oi >= 0 && (bi < 0 || ranks_before(ov, oi, bv, bi))) {
        bv = ov;
        bi = oi;
        bq = oq;
      }
    }
    sel[j] = bi;
    selv[j] = bv;
    if (bq >= 0 && (bq & 31) == lane) taken |= 1u << (bq >> 5);
  }
  write_slots_and_gates(sel, selv, k, topk_idx + (size_t)t * k, gates + (size_t)t * k, lane);
}

// Tiled recompute of the candidates' chunk sums.  One CTA per (chunk c,
// tile of kCertTT tokens): the tile's h slices and the chunk-c slices of
// the union of its tokens' candidate experts are staged in shared memory,
// each row copied by one warp in coalesced 16-byte pieces (an expert slice serves every token of the tile that has it as a
// candidate); then each (token, candidate) pair is summed by one thread from
// +0 in ascending index with fma.  Pairs are bucketed by expert so that a
// pass over kCertWRows staged experts covers a contiguous run of pairs.
// part[(t * C + c) * kCertQ + q] receives the chunk sum.
__global__ void __launch_bounds__(256, 3) cert_chunk_kernel(
    const uint16_t* __restrict__ h, const uint16_t* __restrict__ wgT, const int32_t* __restrict__ cand,
    const int32_t* __restrict__ ccount, int T, int H, float* __restrict__ part) {
  pdl_wait();      // earlier kernels' outputs are visible from here on
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t csm[];
  uint8_t* s_h = csm;                          // [kCertTT][kCertRow]
  uint8_t* s_w = csm + kCertTT * kCertRow;     // [kCertWRows][kCertRow]
  __shared__ int s_cand[kCertTT * kCertQ];     // the tile's candidate lists
  __shared__ int s_pair[kCertTT * kCertQ];     // union position << 12 | token << 5 | slot, by expert
  __shared__ int s_pos[256];                   // expert -> union position
  __shared__ int s_uexp[256];                  // union position -> expert
  __shared__ int s_ubeg[257];                  // union position -> first pair
  __shared__ int s_ucur[256];
  __shared__ int s_cnt[kCertTT];
  __shared__ int s_nu;
  const int C = (H + kRouterChunk - 1) / kRouterChunk;
  const int c = blockIdx.x, t0 = blockIdx.y * kCertTT;
  const int i0 = c * kRouterChunk, len = min(H - i0, kRouterChunk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nt = min(kCertTT, T - t0);
  const bool piece = lane * 8 < len;   // this lane's 16-byte piece of a slice (len % 128 == 0)
  if (piece)
    for (int r = warp; r < nt; r += 8)
      cp_async_16(s_h + r * kCertRow + 16 * lane, h + (size_t)(t0 + r) * H + i0 + 8 * lane);
  asm volatile("cp.async.commit_group;" ::: "memory");
  for (int e = tid; e < 256; e += blockDim.x) s_ucur[e] = 0;
  if (tid < kCertTT) s_cnt[tid] = tid < nt ? max(ccount[t0 + tid], 0) : 0;   // -1: finished by the filter
  __syncthreads();
  for (int p = tid; p < kCertTT * kCertQ; p += blockDim.x) {
    const int r = p / kCertQ, q = p % kCertQ;
    if (q < s_cnt[r]) {
      const int e = cand[(size_t)(t0 + r) * kCertQ + q];
      s_cand[p] = e;
      atomicAdd(&s_ucur[e], 1);
    }
  }
  __syncthreads();
  if (warp == 0) {
    // union positions in ascending expert order and each expert's first pair
    // (lane l handles experts 8l .. 8l+7)
    int pc[8], flag = 0, pairs = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      pc[j] = s_ucur[lane * 8 + j];
      flag += pc[j] > 0;
      pairs += pc[j];
    }
    int fi = flag, pi = pairs;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int fo = __shfl_up_sync(0xffffffffu, fi, off), po = __shfl_up_sync(0xffffffffu, pi, off);
      if (lane >= off) {
        fi += fo;
        pi += po;
      }
    }
    int u = fi - flag, pb = pi - pairs;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane * 8 + j;
      if (pc[j] > 0) {
        s_uexp[u] = e;
        s_ubeg[u] = pb;
        s_pos[e] = u;
        ++u;
        pb += pc[j];
      }
      s_ucur[e] = 0;
    }
    if (lane == 31) {
      s_nu = fi;
      s_ubeg[fi] = pi;
    }
  }
  __syncthreads();
  for (int p = tid; p < kCertTT * kCertQ; p += blockDim.x) {
    const int r = p / kCertQ, q = p % kCertQ;
    if (q < s_cnt[r]) {
      const int u = s_pos[s_cand[p]];
      s_pair[s_ubeg[u] + atomicAdd(&s_ucur[u], 1)] = (u << 12) | (r << 5) | q;
    }
  }
  const int nu = s_nu;
  for (int u0 = 0; u0 < nu; u0 += kCertWRows) {
    const int nb = min(kCertWRows, nu - u0);
    __syncthreads();   // the pair list is complete / the previous pass is done with s_w
    if (piece)
      for (int r = warp; r < nb; r += 8)
        cp_async_16(s_w + r * kCertRow + 16 * lane, wgT + (size_t)s_uexp[u0 + r] * H + i0 + 8 * lane);
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    const int pend = s_ubeg[u0 + nb];
    for (int pi = s_ubeg[u0] + tid; pi < pend; pi += blockDim.x) {
      const int pr = s_pair[pi];
      const int r = (pr >> 5) & 127, q = pr & 31;
      const uint8_t* hr = s_h + r * kCertRow;
      const uint8_t* wr = s_w + ((pr >> 12) - u0) * kCertRow;
      float acc = 0.0f;
#pragma unroll 4
      for (int i = 0; i < len; i += 8) {
        const uint4 hv = *reinterpret_cast<const uint4*>(hr + 2 * i);
        const uint4 wv = *reinterpret_cast<const uint4*>(wr + 2 * i);
        acc = fmaf(bf16_lo(hv.x), bf16_lo(wv.x), acc);
        acc = fmaf(bf16_hi(hv.x), bf16_hi(wv.x), acc);
        acc = fmaf(bf16_lo(hv.y), bf16_lo(wv.y), acc);
        acc = fmaf(bf16_hi(hv.y), bf16_hi(wv.y), acc);
        acc = fmaf(bf16_lo(hv.z), bf16_lo(wv.z), acc);
        acc = fmaf(bf16_hi(hv.z), bf16_hi(wv.z), acc);
        acc = fmaf(bf16_lo(hv.w), bf16_lo(wv.w), acc);
        acc = fmaf(bf16_hi(hv.w), bf16_hi(wv.w), acc);
      }
      part[((size_t)(t0 + r) * C + c) * kCertQ + q] = acc;
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");   // a tile without pairs
}

// Canonical logits of the candidates (chunk sums added to +0 in ascending
// chunk order, then the bias), then top-k and gates: one warp per token,
// lane q holds candidate q.  Tokens the filter finished are skipped.
__global__ void __launch_bounds__(256) cert_finalize_kernel(
    const float* __restrict__ part, const int32_t* __restrict__ cand, const int32_t* __restrict__ ccount,
    const float* __restrict__ bias, int T, int C, int k, int32_t* __restrict__ topk_idx,
    float* __restrict__ gates) {
  pdl_wait();      // earlier kernels' outputs are visible from here on
  pdl_trigger();
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const int nc = ccount[t];
  if (nc < 0) return;
  const bool mine = lane < nc;
  int e = -1;
  float cv = 0.0f;
  if (mine) {
    e = cand[(size_t)t * kCertQ + lane];
    const float* pp = part + (size_t)t * C * kCertQ + lane;
    float total = 0.0f;
    for (int c0 = 0; c0 < C; c0 += 8) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = c0 + j < C ? pp[(size_t)(c0 + j) * kCertQ] : 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (c0 + j < C) total = total + v[j];
    }
    cv = bias ? total + bias[e] : total;
  }
  // sort the candidates best first, keyed by their position q (the list is in
  // ascending expert order, so q breaks ties like the expert index); the
  // first k positions are the selection, written in expert order
  float sv = cv;
  int sq = mine ? lane : -1;
  sel::warp_sort_best_first(sv, sq, lane);
  const unsigned chosen = __reduce_or_sync(full, (lane < k && sq >= 0) ? 1u << sq : 0u);
  sel::write_gates_lanes(chosen, e, cv, lane, topk_idx + (size_t)t * k, gates + (size_t)t * k);
}

}  // namespace

void launch_gate_prep(const uint16_t* w_gate, uint16_t* wgT, float* norm_w, int H, int N,
                      cudaStream_t s) {
  const int tblocks = ((N + 31) / 32) * ((H + 31) / 32);
  launch_pdl(gate_prep_kernel, dim3(tblocks + N / 8), dim3(256), 0, s, w_gate, wgT, norm_w, H, N, tblocks);
}

float router_cert_beta(int H) {
  const int chunks = (H + kRouterChunk - 1) / kRouterChunk;
  return (float)((H / 16 + 1) * 0x1p-20 + (kRouterChunk + chunks + 1) * 0x1p-24);
}

bool route_certified_ok(int H) { return H <= kCertMaxH; }

size_t route_certified_scratch_floats(int T, int H) {
  const size_t C = (size_t)(H + kRouterChunk - 1) / kRouterChunk;
  return (size_t)T * C * kCertQ + (size_t)T * kCertQ + (size_t)T;
}

void launch_route_certified(const float* logits_tc, const float* bias, const uint16_t* h,
                            const uint16_t* wgT, const float* norm_w, int T, int H, int N, int k,
                            int32_t* topk_idx, float* gates, int32_t* n_cand, float* scratch,
                            cudaStream_t s) {
  const int C = (H + kRouterChunk - 1) / kRouterChunk;
  float* part = scratch;
  int32_t* cand = reinterpret_cast<int32_t*>(scratch + (size_t)T * C * kCertQ);
  int32_t* ccount = cand + (size_t)T * kCertQ;
  launch_pdl(route_certified_kernel, dim3((T + kCertWarps - 1) / kCertWarps), dim3(kCertWarps * 32), 0, s,
             logits_tc, bias, h, wgT, norm_w, T, H, N, k, router_cert_beta(H), topk_idx, gates, n_cand, cand,
             ccount);
  const size_t smem = (size_t)(kCertTT + kCertWRows) * kCertRow;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaFuncSetAttribute(cert_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  launch_pdl(cert_chunk_kernel, dim3(C, (T + kCertTT - 1) / kCertTT), dim3(256), smem, s, h, wgT,
             (const int32_t*)cand, (const int32_t*)ccount, T, H, part);
  launch_pdl(cert_finalize_kernel, dim3((T + 7) / 8), dim3(256), 0, s, (const float*)part,
             (const int32_t*)cand, (const int32_t*)ccount, bias, T, C, k, topk_idx, gates);
}

// The chunked router: for a few tokens always (many CTAs share the weight
// reads of a decode step), and for batches whose router work T * H * N is
// at most 3 * 2^28 multiply-adds; above that the certified tensor-core
// router, whose cost grows with T * H (measured crossings: the Qwen-like
// router near T = 2800, 0.053 ms either way at 2048 and 0.089 chunked
// against 0.071 at 4096; the DeepSeek-like one near T = 600, 0.132 against
// 0.099 at 1024).  Every path gives the same bits.
// The caller's path flags may force one path where the tensor-core router
// can serve the call (the tests compare the two).
constexpr long long kChunkedRouterMaxWork = 3ll << 28;

bool chunked_router_ok(int T, int H, int N, bool tc_router, uint32_t path_flags) {
  if (!tc_router) return true;
  if (path_flags & kPathRouterTc) return false;
  if (path_flags & kPathRouterChunked) return true;
  if (T <= kDecodeRouterMaxT) return true;
  return (long long)T * H * N <= kChunkedRouterMaxWork;
}

size_t chunked_router_part_floats(int T, int H, int N) {
  const int chunks = (H + kRouterChunk - 1) / kRouterChunk;
  return (size_t)T * chunks * N;
}

template <int LE, int TQ, int EQ = 1>
void launch_partials(const uint16_t* h, const uint16_t* w_gate, float* part, int T, int H, int N, bool vec,
                     cudaStream_t s) {
  constexpr int TB = kPartWarps * (32 / (LE / EQ)) * TQ;
  const int chunks = (H + kRouterChunk - 1) / kRouterChunk;
  const dim3 grid((unsigned)chunks, (unsigned)((N + LE - 1) / LE), (unsigned)((T + TB - 1) / TB));
  const size_t smem = sizeof(uint16_t) * ((size_t)kRouterChunk * LE + (size_t)TB * kPartRow);
  auto kernel = vec ? router_partials_kernel<true, LE, TQ, EQ> : router_partials_kernel<false, LE, TQ, EQ>;
  static bool attr_set[64][2] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev][vec ? 1 : 0]) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (dev >= 0 && dev < 64) attr_set[dev][vec ? 1 : 0] = true;
  }
  launch_pdl(kernel, dim3(grid), dim3(kPartWarps * 32), smem, s, h, w_gate, T, H, N, part);
}

void launch_router_partials(const uint16_t* h, const uint16_t* w_gate, float* part, int T, int H, int N,
                            cudaStream_t s) {
  const bool vec = N % 8 == 0 && H % 8 == 0 && (reinterpret_cast<uintptr_t>(w_gate) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(h) & 15u) == 0;
  // a few tokens: one token per thread (more CTAs); batches: four
  const bool few = T <= kDecodeRouterMaxT;
  if (N <= 8) {
    if (few) launch_partials<8, 1>(h, w_gate, part, T, H, N, vec, s);
    else launch_partials<8, 4>(h, w_gate, part, T, H, N, vec, s);
  } else if (N <= 16) {
    if (few) launch_partials<16, 1>(h, w_gate, part, T, H, N, vec, s);
    else launch_partials<16, 4>(h, w_gate, part, T, H, N, vec, s);
  } else {
    // batches: 4 experts x 4 tokens per thread (16 chains; 8-byte weight
    // loads, token pairs per 4-byte load)
    if (few) launch_partials<32, 1>(h, w_gate, part, T, H, N, vec, s);
    else launch_partials<32, 4, 4>(h, w_gate, part, T, H, N, vec, s);
  }
}

void launch_router_chunked(const uint16_t* h, const uint16_t* w_gate, const float* bias, float* part,
                           float* logits, int32_t* topk_idx, float* gates, int T, int H, int N, int k,
                           cudaStream_t s) {
  const int chunks = (H + kRouterChunk - 1) / kRouterChunk;
  launch_router_partials(h, w_gate, part, T, H, N, s);
  launch_pdl(router_reduce_kernel, dim3(T), dim3((N + 31) / 32 * 32), 0, s, part, bias, T, N, chunks, k, logits, topk_idx, gates);
}

}  // namespace moe
