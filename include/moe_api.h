/*
 * moe_api.h - C ABI of the batch-invariant Mixture-of-Experts layer forward
 * for NVIDIA GB300 (sm_103a).  Library: libmoe_gb300.so.
 *
 * The layer, per token h (row of h [T, H]):
 *   logits = h . W_g (+ bias)                          router, N scores
 *   experts, gates = top-k of softmax(logits), renormalised over the k
 *   capacity check per expert (overflowing routes are dropped)
 *   out = h + sum over kept routes of gate * SwiGLU_e(h)  (+ shared expert)
 * as stated in "Mixture-of-Experts Routing at Inference Time" (ACE Journal),
 * section "How sparse routing works", Figure 1, and "The hard part: token
 * dropping is a silent correctness bug", Figure 2; and in "Mixture-of-experts
 * routing and LLM repeatability" (the per-token pseudo-code, the Switch
 * capacity rule).  The split into route -> dispatch/align -> expert FFN ->
 * combine follows Figure 3 of the first page (router top-k, capacity check
 * and overflow policy, expert compute).
 *
 * Batch invariance ("Why temperature=0 Still Gives Different Answers: Batch
 * Invariance", section "What is batch invariance in LLM inference?"): every
 * reduction has one fixed split and order regardless of T, with no split-K
 * and no atomics, so a token's outputs are bitwise identical regardless of the
 * other tokens of the batch and whichever padded block its routes land in.  The only
 * exception is the capacity rule itself, which couples tokens by design.
 *
 * Conventions for every entry point:
 *   - Pointers are device memory owned by the caller unless the name says
 *     _host.  The library allocates no device memory; scratch comes from the
 *     caller's workspace `ws` of `ws_bytes` bytes (see moe_workspace_bytes).
 *   - bf16 tensors are passed as uint16_t bit patterns, row-major.
 *   - Every device pointer must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Argument errors are returned synchronously before
 *     anything is launched.  MOE_ERR_CUDA reports a launch error.
 *   - T == 0 is a no-op that returns MOE_OK.
 *   - Device-side anomalies (an expert id outside [0, N) passed in through
 *     moe_dispatch_align, a pipeline wait that timed out) never trap: they set
 *     bits of the device status word held in the workspace, the offending work
 *     is skipped, and moe_get_device_status reports them.
 *   - Routes are numbered r = t*k + j (token t, slot j): the flattened route
 *     identifier of "Route-Block Membership Selects Packed-AWQ Arithmetic",
 *     section "The bookkeeping before the matrix multiplication".
 */
#ifndef MOE_API_H
#define MOE_API_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Layer shape.  Supported: H % 128 == 0, I % 128 == 0, Is % 128 == 0,
 * 1 <= N <= 256, 1 <= k <= min(N, 16), B % 8 == 0 and 8 <= B <= 128 with
 * 128 % B == 0, T <= 1,048,576 and T*k < 2^31. */
typedef struct moe_config {
  int32_t hidden;              /* H */
  int32_t num_experts;         /* N routed experts */
  int32_t top_k;               /* k */
  int32_t intermediate;        /* I, routed expert FFN width */
  int32_t block_size;          /* B, rows per padded expert block */
  float capacity_factor;       /* > 0: capacity ceil(cf*T*k/N) per expert; <= 0: no limit */
  int32_t shared_intermediate; /* Is of the always-on shared expert; 0: none */
} moe_config;

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null or misaligned pointer, negative size, inconsistent sizes */
  MOE_ERR_UNSUPPORTED = 2, /* shape outside the supported set above */
  MOE_ERR_WORKSPACE = 3,   /* workspace smaller than moe_workspace_bytes(cfg, T) */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
  MOE_ERR_DEVICE = 5       /* the device status word is non-zero */
} moe_status;

/* Bits of the device status word. */
#define MOE_DEV_ERR_EXPERT_RANGE 0x1 /* a topk_idx entry outside [0, N): route not dispatched */
#define MOE_DEV_ERR_TIMEOUT 0x2      /* a bounded pipeline wait gave up; outputs are invalid */
#define MOE_DEV_ERR_BAD_BLOCKS 0x4   /* moe_expert_ffn got a block list that is unsorted, out of
                                        range or longer than the bound: no expert work was done */

/* Text for a status code (static storage). */
const char* moe_status_string(moe_status s);

/* Checks a configuration against the supported set. */
moe_status moe_check_config(const moe_config* cfg);

/* Expert capacity for a batch of T tokens: ceil(cf*T*k/N), or -1 (no limit).
 * Capacity per "Mixture-of-experts routing and LLM repeatability" (tokens per
 * expert times a capacity factor), rounded up. */
int32_t moe_capacity(const moe_config* cfg, int32_t T);

/* Upper bounds used to size caller buffers for T tokens:
 *   rows of sorted_route_ids (and of y_perm):  T*k + N*(B-1)
 *   entries of block_expert:                   (T*k)/B + N                */
int64_t moe_max_padded_rows(const moe_config* cfg, int32_t T);
int64_t moe_max_blocks(const moe_config* cfg, int32_t T);

/* Bytes of workspace that every call below needs for up to max_tokens
 * tokens (0 if the configuration is invalid).  The workspace holds the
 * intermediate tensors of moe_forward, the tile list of the grouped GEMMs and
 * the device status word.  Contents need not be initialised; the layout is a
 * fixed function of (cfg, max_tokens), so a call with T <= max_tokens may use
 * any workspace sized for max_tokens. */
size_t moe_workspace_bytes(const moe_config* cfg, int32_t max_tokens);

/* Router: logits, softmax, top-k, renormalised gates ("Mixture-of-Experts
 * Routing at Inference Time", "How sparse routing works" and its TopKRouter).
 *   h        [T, H]  bf16        w_gate [H, N] bf16     router_bias [N] fp32 or NULL
 *   topk_idx [T, k]  int32 out   experts sorted by ascending index
 *   topk_gate[T, k]  fp32  out   exp(l_j - m) / sum_sel exp(l_s - m), m = max selected
 *   logits_out [T, N] fp32 out or NULL
 * Logits are fp32 with a fixed order: H cut into 256-element chunks, each
 * summed from +0 in ascending index, chunk sums added in ascending order to a
 * total starting at +0, bias added last (fixed-chunk reduction of "Why
 * temperature=0 Still Gives Different Answers", Tier 2).  Selection ranks
 * larger logits first, equal logits by lower expert index, NaN last. */
moe_status moe_route(const moe_config* cfg, int32_t T, const uint16_t* h, const uint16_t* w_gate,
                     const float* router_bias, int32_t* topk_idx, float* topk_gate,
                     float* logits_out, void* ws, size_t ws_bytes, void* stream);

/* Router paths.  With logits_out != NULL, when N is not a multiple of 128, or
 * when H > 8192, moe_route computes every logit in the canonical order on CUDA cores.
 * Otherwise (moe_forward, or moe_route without logits_out, N % 128 == 0) it
 * first computes l_tc = h . W_g on the tensor cores, bounds |l_tc - l| by
 * delta_t = beta(H) * ||h_t|| * max_e ||W_g[:,e]|| (+ bias rounding), keeps
 * as candidates the experts with l_tc >= L_k - 2 delta_t (L_k = k-th largest
 * l_tc; all experts if anything is non-finite) and computes canonical logits
 * for those only.  Experts below the cut provably cannot be in the top-k,
 * so topk_idx and topk_gate are bit-identical on both paths.
 *   beta(H) = (H/16 + 1) 2^-20 + (256 + ceil(H/256) + 1) 2^-24 covers
 *   H/16 tensor-core K=16 steps at a relative error of 2^-20 each (several
 *   times the truncation error of a 16-term fp32 block sum) and the fp32
 *   additions of the canonical order. */
float moe_router_cert_beta(int32_t hidden);

/* Diagnostic: the tensor-core logits l_tc = h . W_g [T, N] fp32 (no bias) that
 * the filter uses (MOE_ERR_UNSUPPORTED unless N % 128 == 0).  Not the
 * canonical logits; the router margin and the filter width can be studied
 * with them. */
moe_status moe_router_tc_logits(const moe_config* cfg, int32_t T, const uint16_t* h,
                                const uint16_t* w_gate, float* logits_out, void* ws,
                                size_t ws_bytes, void* stream);

/* Diagnostic: the tensor-core router path of moe_route (same topk_idx and
 * topk_gate), also reporting per token how many experts passed the filter
 * and had their canonical logits computed: n_candidates [T] int32 (k..N).
 * MOE_ERR_UNSUPPORTED unless N % 128 == 0 and H <= 8192. */
moe_status moe_route_filtered(const moe_config* cfg, int32_t T, const uint16_t* h,
                              const uint16_t* w_gate, const float* router_bias, int32_t* topk_idx,
                              float* topk_gate, int32_t* n_candidates, void* ws, size_t ws_bytes,
                              void* stream);

/* Capacity-limited dispatch and stable alignment into padded expert blocks.
 * Input topk_idx [T, k] (from moe_route, or recorded routes to replay).
 * Capacity is filled in batch order: an expert keeps its first C routes by
 * ascending route id; the rest are dropped and ride the residual (Figure 2 of
 * "Mixture-of-Experts Routing at Inference Time").  Stable construction
 * ("Route-Block Membership Selects Packed-AWQ Arithmetic", "Stable
 * construction selected a third trajectory"): for e = 0..N-1, expert e's kept
 * routes in ascending r, padded with the sentinel T*k to a multiple of B.
 * Outputs (device):
 *   route_kept      [T*k]                    uint8, 1 = kept
 *   route_pos       [T*k]                    int32, row in sorted_route_ids, -1 if not kept
 *   sorted_route_ids[moe_max_padded_rows]    int32, first *num_padded rows valid
 *   block_expert    [moe_max_blocks]         int32, first *num_padded/B valid
 *   num_padded      [1] int32,  expert_counts [N] int32 (kept), num_dropped [1] int32
 * Integer results only, no atomics: identical bits on every run. */
moe_status moe_dispatch_align(const moe_config* cfg, int32_t T, const int32_t* topk_idx,
                              uint8_t* route_kept, int32_t* route_pos, int32_t* sorted_route_ids,
                              int32_t* block_expert, int32_t* num_padded, int32_t* expert_counts,
                              int32_t* num_dropped, void* ws, size_t ws_bytes, void* stream);

/* Grouped SwiGLU expert FFN over the padded blocks, on tcgen05 tensor cores:
 *   for every padded row p of expert e = block_expert[p / B] with route r:
 *     x = h[r / k] (zero for the sentinel), [g | u] = x . W13_e,
 *     a = bf16(silu(g) * u), y_perm[p] = a . W2_e  (fp32)
 *   and, when cfg->shared_intermediate > 0, y_shared[t] = SwiGLU_shared(h[t]).
 *   w13 [N, H, 2I] bf16 (gate columns 0..I-1, up columns I..2I-1),
 *   w2 [N, I, H] bf16, w13_shared [H, 2Is], w2_shared [Is, H] (or NULL when
 *   Is == 0); y_perm [moe_max_padded_rows, H] fp32 out; y_shared [T, H] fp32
 *   out or NULL when Is == 0.  Rows of y_perm that hold the sentinel get
 *   x = 0 (so a = 0 and y = 0 for finite weights); rows past *num_padded are
 *   not written.
 * One tile shape and one K order for every T, no split-K: each y row
 * depends only on its own x row and the expert's weights. */
moe_status moe_expert_ffn(const moe_config* cfg, int32_t T, const uint16_t* h, const uint16_t* w13,
                          const uint16_t* w2, const uint16_t* w13_shared,
                          const uint16_t* w2_shared, const int32_t* sorted_route_ids,
                          const int32_t* block_expert, const int32_t* num_padded, float* y_perm,
                          float* y_shared, void* ws, size_t ws_bytes, void* stream);

/* Gate-weighted combine into the residual:
 *   out[t] = bf16( h[t] + sum_{j ascending, kept} topk_gate[t,j] * y_perm[route_pos[t*k+j]]
 *                  + y_shared[t] )
 * accumulated in fp32 in that fixed order.  y_shared may be NULL.  out [T,H] bf16. */
moe_status moe_combine(const moe_config* cfg, int32_t T, const uint16_t* h, const float* topk_gate,
                       const uint8_t* route_kept, const int32_t* route_pos, const float* y_perm,
                       const float* y_shared, uint16_t* out, void* stream);

/* The whole layer: moe_route -> moe_dispatch_align -> moe_expert_ffn ->
 * moe_combine on `stream`, intermediates in the workspace.  No host
 * synchronisation and no device-to-host copy. */
moe_status moe_forward(const moe_config* cfg, int32_t T, const uint16_t* h, const uint16_t* w_gate,
                       const float* router_bias, const uint16_t* w13, const uint16_t* w2,
                       const uint16_t* w13_shared, const uint16_t* w2_shared, uint16_t* out,
                       void* ws, size_t ws_bytes, void* stream);

/* moe_forward with the token rows in host memory: copies h_host [T, H] to the
 * device (into the workspace), runs the layer and copies the result back to
 * out_host [T, H].  Weights stay on the device.  Host buffers should be
 * page-locked for the copies to be asynchronous; the call returns after
 * enqueueing and the caller synchronises `stream` before reading out_host. */
moe_status moe_forward_hostio(const moe_config* cfg, int32_t T, const uint16_t* h_host,
                              const uint16_t* w_gate, const float* router_bias,
                              const uint16_t* w13, const uint16_t* w2,
                              const uint16_t* w13_shared, const uint16_t* w2_shared,
                              uint16_t* out_host, void* ws, size_t ws_bytes, void* stream);

/* moe_forward that also records caller-created CUDA events (cudaEvent_t
 * handles, at least n_events = 8) on `stream` at the stage boundaries:
 *   events[0] before the router          events[4] after the W13 GEMM
 *   events[1] after the router           events[5] after the W2 GEMM
 *   events[2] after dispatch/alignment   events[6] after the shared expert
 *   events[3] after tile list + row gather   events[7] after the combine
 * so the caller can read per-kernel device times (cudaEventElapsedTime)
 * without extra synchronisation.  Same computation and bits as moe_forward. */
moe_status moe_forward_timed(const moe_config* cfg, int32_t T, const uint16_t* h,
                             const uint16_t* w_gate, const float* router_bias, const uint16_t* w13,
                             const uint16_t* w2, const uint16_t* w13_shared,
                             const uint16_t* w2_shared, uint16_t* out, void* ws, size_t ws_bytes,
                             void* const* events, int32_t n_events, void* stream);

/* Number of kernel launches one moe_forward makes for this configuration. */
int32_t moe_forward_launch_count(const moe_config* cfg);

/* moe_dispatch_align for callers that cannot allocate device memory (for
 * example a serving loop whose memory is fixed at start-up, or code running
 * while another framework owns the allocator), so cannot pass a workspace.
 * The pages have no counterpart to this entry point; it is a deployment aid.
 * Same inputs, outputs and bits as moe_dispatch_align, but it allocates
 * nothing: its scratch is one fixed device array inside this library
 * (~321 KB on every GPU that loads it, held until the process exits).
 *   - Limit: T*k <= 65536 routes (and N <= 256); larger batches return
 *     MOE_ERR_UNSUPPORTED without doing anything.
 *   - status_out: device int32 or NULL; receives this call's device status
 *     word (MOE_DEV_ERR_EXPERT_RANGE for expert ids outside [0, N)).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents (the call clears what must start at zero).  Calls that
 *     overlap on the GPU (e.g. on two streams at once) race on it: order them. */
moe_status moe_dispatch_align_noalloc(const moe_config* cfg, int32_t T, const int32_t* topk_idx,
                                      uint8_t* route_kept, int32_t* route_pos,
                                      int32_t* sorted_route_ids, int32_t* block_expert,
                                      int32_t* num_padded, int32_t* expert_counts,
                                      int32_t* num_dropped, int32_t* status_out, void* stream);

/* Reads the device status word of `ws` (synchronises `stream`). */
moe_status moe_get_device_status(const void* ws, int32_t* status_out, void* stream);

/* Clears the device status word of `ws` (asynchronous on `stream`). */
moe_status moe_clear_device_status(void* ws, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_API_H */
