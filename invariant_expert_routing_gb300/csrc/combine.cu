// Gate-weighted combine into the residual stream ("Mixture-of-Experts Routing
// at Inference Time", "How sparse routing works" and Figure 2): each token
// gets h plus its kept experts' outputs scaled by their gates; a route that
// overflowed contributes nothing.
//
// out[t,:] = bf16( h[t,:] + acc ),  acc = fma over kept slots j = 0..S-1 in
// ascending order of gate[t,j] * y_perm[route_pos[t*S+j], :], then + y_shared
// (y_perm and y_shared: the expert GEMMs' fp32 results stored as bf16; the
// sum itself is fp32).
// S is the number of route slots per token: k for token choice, N for expert
// choice (slot e = expert e).  The kept slots are first listed in ascending j
// in shared memory; skipping the others leaves the chain of fmas unchanged.
// With many tokens a CTA takes one row: 8 consecutive features per thread and
// 16-byte accesses when the row is a multiple of 2048 features, else 4.  With few tokens a row is split over gridDim.y CTAs
// (so that a lone token's row is spread over several SMs), 4 consecutive
// features per thread, 64-bit loads of the bf16 y_perm issued eight slots at
// a time before their fmas.  The order of the sum is fixed and independent of
// T and of the grid.
#include <cuda_bf16.h>
#include <cstdint>

#include "kernels.h"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int kMaxSlots = 256;

// Four consecutive bf16 values (8-byte aligned) widened to fp32.
__device__ __forceinline__ float4 load_bf16x4(const uint16_t* p) {
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
  return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                     __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
}

// Eight consecutive bf16 values (16-byte aligned) widened to fp32.
__device__ __forceinline__ void load_bf16x8(const uint16_t* p, float (&v)[8]) {
  const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}

// kForm: 0 many tokens, 4 features per thread; 1 many tokens, 8 features per
// thread (rows of a multiple of 2048 features: every thread has whole
// passes); 2 few tokens, a row split over gridDim.y CTAs.
template <int kForm>
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ h,
                                                      const float* __restrict__ gates,
                                                      const uint8_t* __restrict__ route_kept,
                                                      const int32_t* __restrict__ route_pos,
                                                      const uint16_t* __restrict__ y_perm,
                                                      const uint16_t* __restrict__ y_shared,
                                                      uint16_t* __restrict__ out, int H, int k,
                                                      long long max_rows) {
  pdl_wait();      // earlier kernels' outputs are visible from here on
  const int t = blockIdx.x;
  __shared__ int s_pos[kMaxSlots];
  __shared__ float s_gate[kMaxSlots];
  __shared__ int s_wcnt[8];
  // few tokens: this thread's first h (and y_shared) piece is requested
  // before the slot list is built (it depends on neither)
  const int d_first = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
  uint2 h_first = make_uint2(0u, 0u), ys_first = make_uint2(0u, 0u);
  if (kForm == 2 && d_first < H) {
    h_first = __ldg(reinterpret_cast<const uint2*>(h + (size_t)t * H + d_first));
    if (y_shared) ys_first = __ldg(reinterpret_cast<const uint2*>(y_shared + (size_t)t * H + d_first));
  }
  // list the kept slots in ascending j (k <= 256 = blockDim.x: one slot per thread)
  const int j = threadIdx.x, lane = j & 31, w = j >> 5;
  bool use = false;
  int pos = -1;
  float g = 0.0f;
  if (j < k) {
    const size_t r = (size_t)t * k + j;
    pos = route_pos[r];
    use = route_kept[r] && pos >= 0 && (long long)pos < max_rows;
    g = gates[r];
  }
  const unsigned m = __ballot_sync(0xffffffffu, use);
  if (lane == 0) s_wcnt[w] = __popc(m);
  __syncthreads();
  int before = __popc(m & ((1u << lane) - 1u)), n_used = 0;
  for (int i = 0; i < 8; ++i) {
    if (i < w) before += s_wcnt[i];
    n_used += s_wcnt[i];
  }
  if (use) {
    s_pos[before] = pos;
    s_gate[before] = g;
  }
  __syncthreads();
  if (kForm == 1) {
    // many tokens (one CTA per row): 8 consecutive features per thread,
    // 16-byte loads and stores; occupancy hides the latency.  Each feature's
    // chain of fmas is the one of the split-row form below.
    for (int d = threadIdx.x * 8; d < H; d += blockDim.x * 8) {
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
      for (int i = 0; i < n_used; ++i) {
        const float g = s_gate[i];
        float y[8];
        load_bf16x8(y_perm + (size_t)s_pos[i] * H + d, y);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = fmaf(g, y[q], acc[q]);
      }
      if (y_shared) {
        float ys[8];
        load_bf16x8(y_shared + (size_t)t * H + d, ys);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = acc[q] + ys[q];
      }
      float hv[8];
      load_bf16x8(h + (size_t)t * H + d, hv);
      uint4 ov;
      ov.x = pack_bf16x2(hv[0] + acc[0], hv[1] + acc[1]);
      ov.y = pack_bf16x2(hv[2] + acc[2], hv[3] + acc[3]);
      ov.z = pack_bf16x2(hv[4] + acc[4], hv[5] + acc[5]);
      ov.w = pack_bf16x2(hv[6] + acc[6], hv[7] + acc[7]);
      *reinterpret_cast<uint4*>(out + (size_t)t * H + d) = ov;
    }
    return;
  }
  for (int d = (blockIdx.y * blockDim.x + threadIdx.x) * 4; d < H; d += gridDim.y * blockDim.x * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (kForm == 2) {   // few tokens: eight slots' loads in flight before their fmas
      for (int i0 = 0; i0 < n_used; i0 += 8) {
        float4 y[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (i0 + q < n_used)
            y[q] = load_bf16x4(y_perm + (size_t)s_pos[i0 + q] * H + d);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (i0 + q < n_used) {
            const float g = s_gate[i0 + q];
            acc.x = fmaf(g, y[q].x, acc.x);
            acc.y = fmaf(g, y[q].y, acc.y);
            acc.z = fmaf(g, y[q].z, acc.z);
            acc.w = fmaf(g, y[q].w, acc.w);
          }
        }
      }
    } else {            // many tokens: occupancy hides the latency (fewer registers)
      for (int i = 0; i < n_used; ++i) {
        const float g = s_gate[i];
        const float4 y = load_bf16x4(y_perm + (size_t)s_pos[i] * H + d);
        acc.x = fmaf(g, y.x, acc.x);
        acc.y = fmaf(g, y.y, acc.y);
        acc.z = fmaf(g, y.z, acc.z);
        acc.w = fmaf(g, y.w, acc.w);
      }
    }
    const bool first = kForm == 2 && d == d_first;
    if (y_shared) {
      const float4 ys = first ? make_float4(__uint_as_float(ys_first.x << 16), __uint_as_float(ys_first.x & 0xFFFF0000u),
                                            __uint_as_float(ys_first.y << 16), __uint_as_float(ys_first.y & 0xFFFF0000u))
                              : load_bf16x4(y_shared + (size_t)t * H + d);
      acc.x = acc.x + ys.x;
      acc.y = acc.y + ys.y;
      acc.z = acc.z + ys.z;
      acc.w = acc.w + ys.w;
    }
    const uint2 hv = first ? h_first : __ldg(reinterpret_cast<const uint2*>(h + (size_t)t * H + d));
    const float h0 = __uint_as_float(hv.x << 16), h1 = __uint_as_float(hv.x & 0xFFFF0000u);
    const float h2 = __uint_as_float(hv.y << 16), h3 = __uint_as_float(hv.y & 0xFFFF0000u);
    const __nv_bfloat16 o0 = __float2bfloat16_rn(h0 + acc.x), o1 = __float2bfloat16_rn(h1 + acc.y);
    const __nv_bfloat16 o2 = __float2bfloat16_rn(h2 + acc.z), o3 = __float2bfloat16_rn(h3 + acc.w);
    uint2 ov;
    ov.x = (uint32_t)__bfloat16_as_ushort(o0) | ((uint32_t)__bfloat16_as_ushort(o1) << 16);
    ov.y = (uint32_t)__bfloat16_as_ushort(o2) | ((uint32_t)__bfloat16_as_ushort(o3) << 16);
    *reinterpret_cast<uint2*>(out + (size_t)t * H + d) = ov;
  }
}

// The same combine with one warp per token (many tokens, at most 16 slots):
// no block barriers, so the next token's slot list is requested while other
// warps' rows are in flight.  Lane j < S holds slot j's route; the kept slots,
// in ascending j, are broadcast from their lanes; each lane then forms 8
// consecutive features per step (16-byte accesses), the kept slots' rows
// requested (eight at a time) before their fmas, in the order of the forms
// above.
constexpr int kWarpMaxSlots = 16;

__global__ void __launch_bounds__(256) combine_warp_kernel(const uint16_t* __restrict__ h,
                                                           const float* __restrict__ gates,
                                                           const uint8_t* __restrict__ route_kept,
                                                           const int32_t* __restrict__ route_pos,
                                                           const uint16_t* __restrict__ y_perm,
                                                           const uint16_t* __restrict__ y_shared,
                                                           uint16_t* __restrict__ out, int T, int H, int k,
                                                           long long max_rows) {
  pdl_wait();      // earlier kernels' outputs are visible from here on
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  bool use = false;
  int pos = -1;
  float g = 0.0f;
  if (lane < k) {
    const size_t r = (size_t)t * k + lane;
    pos = route_pos[r];
    use = route_kept[r] && pos >= 0 && (long long)pos < max_rows;
    g = gates[r];
  }
  const unsigned m = __ballot_sync(0xffffffffu, use);
  const int nu = __popc(m);
  // the u-th kept slot's row and gate, for u < nu (ascending slot order)
  int rows_u[kWarpMaxSlots];
  float g_u[kWarpMaxSlots];
  {
    unsigned mm = m;
#pragma unroll
    for (int u = 0; u < kWarpMaxSlots; ++u) {
      const int src = mm ? __ffs(mm) - 1 : 0;
      rows_u[u] = __shfl_sync(0xffffffffu, pos, src);
      g_u[u] = __shfl_sync(0xffffffffu, g, src);
      mm &= mm - 1u;
    }
  }
  const int chunks = H / 8;
  const size_t trow = (size_t)t * H;
  for (int c = lane; c < chunks; c += 32) {
    const size_t col = (size_t)c * 8;
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
    for (int u0 = 0; u0 < kWarpMaxSlots; u0 += 8) {
      if (u0 < nu) {
        uint4 raw[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (u0 + u < nu) raw[u] = __ldg(reinterpret_cast<const uint4*>(y_perm + (size_t)rows_u[u0 + u] * H + col));
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (u0 + u < nu) {
            const float gi = g_u[u0 + u];
            const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc[2 * q] = fmaf(gi, __uint_as_float(w[q] << 16), acc[2 * q]);
              acc[2 * q + 1] = fmaf(gi, __uint_as_float(w[q] & 0xFFFF0000u), acc[2 * q + 1]);
            }
          }
        }
      }
    }
    if (y_shared) {
      float ys[8];
      load_bf16x8(y_shared + trow + col, ys);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = acc[q] + ys[q];
    }
    float hv[8];
    load_bf16x8(h + trow + col, hv);
    uint4 ov;
    ov.x = pack_bf16x2(hv[0] + acc[0], hv[1] + acc[1]);
    ov.y = pack_bf16x2(hv[2] + acc[2], hv[3] + acc[3]);
    ov.z = pack_bf16x2(hv[4] + acc[4], hv[5] + acc[5]);
    ov.w = pack_bf16x2(hv[6] + acc[6], hv[7] + acc[7]);
    *reinterpret_cast<uint4*>(out + trow + col) = ov;
  }
}

}  // namespace

void launch_combine(const uint16_t* h, const float* gates, const uint8_t* route_kept,
                    const int32_t* route_pos, const uint16_t* y_perm, const uint16_t* y_shared,
                    uint16_t* out, int T, int H, int k, int64_t max_rows, cudaStream_t s) {
  // enough CTAs for about two per SM, at most one per 1024 features of a row
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int per_row = (H + 1023) / 1024;
  const int want = T > 0 ? (2 * (sms > 0 ? sms : 1) + T - 1) / T : 1;
  const dim3 grid((unsigned)T, (unsigned)(want < per_row ? (want > 0 ? want : 1) : per_row));
  // a warp per token where a token has several slots and the batch is large
  // (measured: 0.0685 -> 0.062 ms on the Qwen-like T = 8192 combine, 0.435 ->
  // 0.390 ms on the DeepSeek-like T = 16448; slower with two slots or a few
  // hundred tokens, whose warps have too little in flight)
  if (grid.y == 1 && k >= 4 && k <= kWarpMaxSlots && T >= 2048) {
    launch_pdl(combine_warp_kernel, dim3((unsigned)((T + 7) / 8)), dim3(256), 0, s, h, gates, route_kept, route_pos,
               y_perm, y_shared, out, T, H, k, (long long)max_rows);
    return;
  }
  if (grid.y > 1)
    launch_pdl(combine_kernel<2>, dim3(grid), dim3(256), 0, s, h, gates, route_kept, route_pos, y_perm, y_shared,
               out, H, k, (long long)max_rows);
  else if (H % 2048 == 0)
    launch_pdl(combine_kernel<1>, dim3(grid), dim3(256), 0, s, h, gates, route_kept, route_pos, y_perm, y_shared,
               out, H, k, (long long)max_rows);
  else
    launch_pdl(combine_kernel<0>, dim3(grid), dim3(256), 0, s, h, gates, route_kept, route_pos, y_perm, y_shared,
               out, H, k, (long long)max_rows);
}

}  // namespace moe
