/*
 * Seeded synthetic input generator (host side).
 *
 * This module only produces numbers; it holds none of the MoE layer's
 * arithmetic.  The same generator exists as a CUDA kernel in synth_gpu.cu and
 * the two are required to agree bit for bit, so that inputs generated on the
 * device (the 22 GB expert tensors of the large layers) equal the inputs the
 * host-side checker regenerates for itself.
 *
 * Definition (both sides):
 *   mix(x)      = SplitMix64 output function (Steele, Lea and Flood, "Fast
 *                 splittable pseudorandom number generators", OOPSLA 2014):
 *                 z = x + 0x9E3779B97F4A7C15;
 *                 z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9;
 *                 z = (z ^ (z >> 27)) * 0x94D049BB133111EB;
 *                 return z ^ (z >> 31);
 *   stream      = mix(mix(seed) ^ tensor_id)
 *   word(i, w)  = mix(stream + 3*i + w)            (w = 0, 1, 2)
 *   normal(i)   = sum of the twelve 16-bit lanes of word(i,0..2), minus
 *                 393210 (= 12 * 32767.5, rounded): an Irwin-Hall(12)
 *                 approximation of N(0, 65536^2), exact in int32
 *   value(i)    = bf16_rne( (float)normal(i) * scale ),  scale = fp32(std/65536)
 *   uniform(i)  = mix(stream + i)                     (raw 64-bit draw)
 *
 * Every step is integer arithmetic or one IEEE fp32 multiply, so host and
 * device produce identical bits.  Tails are bounded at about 6 sigma.
 */
#include <stdint.h>
#include <string.h>
#include <pthread.h>

static inline uint64_t mix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_stream(uint64_t seed, uint64_t tensor_id) {
  return mix64(mix64(seed) ^ tensor_id);
}

static inline int32_t lanes_sum(uint64_t w) {
  return (int32_t)(w & 0xFFFF) + (int32_t)((w >> 16) & 0xFFFF) +
         (int32_t)((w >> 32) & 0xFFFF) + (int32_t)(w >> 48);
}

static inline int32_t normal_int(uint64_t stream, uint64_t i) {
  uint64_t base = stream + 3 * i;
  return lanes_sum(mix64(base)) + lanes_sum(mix64(base + 1)) + lanes_sum(mix64(base + 2)) - 393210;
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

typedef struct {
  uint16_t* out;
  uint64_t begin, end, offset, stream;
  float scale;
} fill_job;

static void* fill_worker(void* p) {
  fill_job* j = (fill_job*)p;
  for (uint64_t i = j->begin; i < j->end; ++i) {
    float v = (float)normal_int(j->stream, j->offset + i) * j->scale;
    j->out[i] = f32_to_bf16_rne(v);
  }
  return 0;
}

/* Fill out[0..n) with value(offset + i) of stream (seed, tensor_id). */
void synth_normal_bf16(uint16_t* out, uint64_t n, uint64_t offset, uint64_t seed,
                       uint64_t tensor_id, float scale, int nthreads) {
  uint64_t stream = synth_stream(seed, tensor_id);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 64) nthreads = 64;
  if (n < (1u << 16)) nthreads = 1;
  pthread_t th[64];
  fill_job jobs[64];
  uint64_t per = (n + (uint64_t)nthreads - 1) / (uint64_t)nthreads;
  for (int t = 0; t < nthreads; ++t) {
    uint64_t b = per * (uint64_t)t, e = b + per;
    if (b > n) b = n;
    if (e > n) e = n;
    jobs[t].out = out; jobs[t].begin = b; jobs[t].end = e;
    jobs[t].offset = offset; jobs[t].stream = stream; jobs[t].scale = scale;
  }
  int created[64] = {0};
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[t], 0, fill_worker, &jobs[t]) == 0) created[t] = 1;
    else fill_worker(&jobs[t]);
  }
  fill_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t)
    if (created[t]) pthread_join(th[t], 0);
}

/* Raw 64-bit draws uniform(offset + i), i in [0, n). */
void synth_uniform_u64(uint64_t* out, uint64_t n, uint64_t offset, uint64_t seed, uint64_t tensor_id) {
  uint64_t stream = synth_stream(seed, tensor_id);
  for (uint64_t i = 0; i < n; ++i) out[i] = mix64(stream + offset + i);
}
