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

/* Overflow policy for routes past an expert's capacity ("Mixture-of-Experts
 * Routing at Inference Time", Figure 2): drop (the route adds nothing; the
 * token keeps its residual and its other routes) or reroute (the route moves
 * to the token's best-ranked expert that still has room and that the token
 * does not use yet; it keeps its slot's gate). */
#define MOE_OVERFLOW_DROP 0
#define MOE_OVERFLOW_REROUTE 1
/* Routing: token choice (each token takes its top-k experts) or expert choice
 * (each expert takes its top-C tokens of the batch by softmax probability;
 * "Mixture-of-experts routing and LLM repeatability"). */
#define MOE_ROUTING_TOKEN_CHOICE 0
#define MOE_ROUTING_EXPERT_CHOICE 1

/* Layer shape.  Supported: H % 128 == 0, I % 128 == 0, Is % 128 == 0,
 * 1 <= N <= 256, 1 <= k <= min(N, 16), B % 8 == 0 and 8 <= B <= 128 with
 * 128 % B == 0, T <= 1,048,576 and T*S < 2^31, S = route slots per token
 * (k for token choice, N for expert choice).  Zero-initialise the struct:
 * zero is the default of every field. */
typedef struct moe_config {
  int32_t hidden;              /* H */
  int32_t num_experts;         /* N routed experts */
  int32_t top_k;               /* k (expert choice: average experts per token) */
  int32_t intermediate;        /* I, routed expert FFN width */
  int32_t block_size;          /* B, rows per padded expert block */
  double capacity_factor;      /* > 0: capacity ceil(cf*T*k/N) per expert, in fp64 as
                                  ceil(((cf*T)*k)/N); <= 0: no limit (expert choice:
                                  cf = 1, capacity clipped to T) */
  int32_t shared_intermediate; /* Is of the always-on shared expert; 0: none */
  int32_t overflow_policy;     /* MOE_OVERFLOW_DROP or MOE_OVERFLOW_REROUTE (token choice) */
  int32_t routing;             /* MOE_ROUTING_TOKEN_CHOICE or MOE_ROUTING_EXPERT_CHOICE */
  /* Testing and diagnosis only; leave zero in production.  None of these
   * changes a result bit: each forces one of several equivalent ways of
   * computing the same integers and floats, or shortens the bounded waits. */
  uint32_t debug_flags;        /* MOE_DEBUG_* bits */
  int32_t debug_grid_ctas;     /* > 0: at most this many CTAs run the reroute's grid-wide
                                  rounds (more routes per CTA); 0: one per SM */
  int64_t debug_wait_ns;       /* > 0: every bounded device wait gives up after this many ns
                                  (the grouped GEMM's pipeline waits, default 2 s, and the
                                  reroute's grid barrier, default 0.2 s); 0: the defaults */
} moe_config;

/* debug_flags bits.  Each pair of alternatives computes the same bits; a
 * flag only selects which kernels run (the tests compare them). */
#define MOE_DEBUG_ROUTER_TC 0x1u          /* tensor-core router with the certified filter
                                             wherever it can serve the call (N % 128 == 0,
                                             no logits_out), whatever T */
#define MOE_DEBUG_ROUTER_CHUNKED 0x2u     /* chunked CUDA-core router for every batch */
#define MOE_DEBUG_ROW_GATHER 0x4u         /* routed token rows copied in segment order */
#define MOE_DEBUG_ROW_SCATTER 0x8u        /* routed token rows copied token by token
                                             (moe_forward; moe_expert_ffn always gathers) */
#define MOE_DEBUG_NO_DECODE_FRONT 0x10u   /* no fused decode front for T <= 2 */
#define MOE_DEBUG_REROUTE_SEQUENTIAL 0x20u /* reroute: the sequential kernel alone */
#define MOE_DEBUG_REROUTE_GRID 0x40u      /* reroute: grid-wide acceptance rounds for any batch */
#define MOE_DEBUG_REROUTE_ONE_CTA 0x80u   /* reroute: one-CTA acceptance rounds for any batch */
#define MOE_DEBUG_ROUTER_TILE128 0x100u   /* tensor-core router logits in 128-row token tiles */
#define MOE_DEBUG_ROUTER_TILE64 0x200u    /* tensor-core router logits in 64-row token tiles */
#define MOE_DEBUG_SHARED_SERIAL 0x400u    /* moe_forward: the shared expert on the caller's stream after
                                             the routed GEMMs instead of on a second stream */
#define MOE_DEBUG_W13_PAIR 0x800u         /* routed W13 on CTA pairs (the default wherever the
                                             intermediate size is a multiple of 128) */
#define MOE_DEBUG_W2_WIDE 0x1000u         /* routed W2 pairs in wide items (two 256-feature groups per
                                             token tile) whatever the reduction length */
#define MOE_DEBUG_W13_SINGLE 0x2000u      /* routed W13 on single CTAs (M = 128 features x N = 128
                                             token rows, gate and up MMAs per K step) */

/* Output of moe_routing_stats (device memory, 40 bytes). */
typedef struct moe_route_stats {
  int32_t max_expert_load;  /* routes naming the busiest expert */
  int32_t min_expert_load;  /* routes naming the idlest expert */
  int32_t capacity;         /* probe capacity floor(mean load * capacity_factor) */
  int32_t dropped_tokens;   /* sum over experts of max(0, load - capacity) */
  int32_t total_routes;     /* routes with an expert id in [0, N) */
  int32_t reserved;         /* 0 */
  double imbalance_ratio;   /* max load / mean load */
  double drop_fraction;     /* dropped_tokens / total_routes */
} moe_route_stats;

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null or misaligned pointer, negative size, inconsistent sizes */
  MOE_ERR_UNSUPPORTED = 2, /* shape outside the supported set above */
  MOE_ERR_WORKSPACE = 3,   /* workspace smaller than moe_workspace_bytes(cfg, T) */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
  MOE_ERR_DEVICE = 5       /* the device status word has an error bit set */
} moe_status;

/* Bits of the device status word. */
#define MOE_DEV_ERR_EXPERT_RANGE 0x1 /* a topk_idx entry outside [0, N): route not dispatched */
#define MOE_DEV_ERR_TIMEOUT 0x2      /* a bounded pipeline wait gave up; outputs are invalid */
#define MOE_DEV_ERR_BAD_BLOCKS 0x4   /* moe_expert_ffn got a block list that is unsorted, out of
                                        range or longer than the bound: no expert work was done */
/* Informational bit (not an error; moe_get_device_status still returns
 * MOE_OK when it is the only bit set): the reroute's grid-wide acceptance
 * rounds gave up at a device-wide barrier that waited past its limit, and the
 * sequential kernel computed the assignment instead (valid results). */
#define MOE_DEV_NOTE_REROUTE_FALLBACK 0x100
#define MOE_DEV_ERR_MASK 0xFF        /* bits that mark invalid outputs */

/* Text for a status code (static storage). */
const char* moe_status_string(moe_status s);

/* Checks a configuration against the supported set. */
moe_status moe_check_config(const moe_config* cfg);

/* Expert capacity for a batch of T tokens: ceil(cf*T*k/N), or -1 (no limit).
 * Capacity per "Mixture-of-experts routing and LLM repeatability" (tokens per
 * expert times a capacity factor), rounded up.  Expert choice: the tokens
 * each expert takes, min(ceil(cf*T*k/N), T) with cf = 1 when cf <= 0. */
int32_t moe_capacity(const moe_config* cfg, int32_t T);

/* Upper bounds used to size caller buffers for T tokens:
 *   rows of sorted_route_ids (and of y_perm):  T*k + N*(B-1)
 *   entries of block_expert:                   (T*k)/B + N
 * Expert choice: N*P rows and N*P/B blocks exactly, P = moe_capacity rounded
 * up to a multiple of B. */
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

/* The router logits alone: logits_out [T, N] fp32, every expert, in the
 * fixed order of moe_route (CUDA cores).  Input of expert-choice routing,
 * overflow reroute and the router margin. */
moe_status moe_router_logits(const moe_config* cfg, int32_t T, const uint16_t* h,
                             const uint16_t* w_gate, const float* router_bias, float* logits_out,
                             void* ws, size_t ws_bytes, void* stream);

/* Router paths.  With logits_out != NULL, when N is not a multiple of 128,
 * when H > 8192, for at most 64 tokens, or when T * H * N <= 3 * 2^28,
 * moe_route computes every logit in the canonical order on CUDA cores (the
 * chunked router: 256-element chunk sums in parallel CTAs, then an in-order
 * reduce with the top-k; two launches).
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
/* One shard of a capacity-limited batch split across GPUs (or calls) in
 * token order: the same dispatch as moe_dispatch_align on the whole batch of
 * global_tokens tokens, restricted to this shard's routes.  The capacity is
 * C = moe_capacity(cfg, global_tokens); expert_offset [N] int32 (device; NULL
 * for the first shard) holds the routes each expert received in all earlier
 * shards (their moe_routing_stats expert_load, summed), so the shard's routes
 * to expert e keep what the earlier ones left: a route is kept iff its rank
 * among the shard's routes to e is below max(0, C - expert_offset[e]) — the
 * batch-order priority of the unsharded batch ("Mixture-of-Experts Routing
 * at Inference Time": capacity filled in batch order).  Obtaining
 * expert_offset takes one exchange of N integers per shard (an all-gather in
 * rank order); the layout, GEMMs and combine stay local.  Outputs as
 * moe_dispatch_align (this shard's routes and layout; num_dropped counts the
 * shard's dropped routes).  Drop policy and token choice only
 * (MOE_ERR_INVALID_ARG otherwise, or when global_tokens < T). */
moe_status moe_dispatch_align_shard(const moe_config* cfg, int32_t T, int32_t global_tokens,
                                    const int32_t* topk_idx, const int32_t* expert_offset,
                                    uint8_t* route_kept, int32_t* route_pos, int32_t* sorted_route_ids,
                                    int32_t* block_expert, int32_t* num_padded, int32_t* expert_counts,
                                    int32_t* num_dropped, void* ws, size_t ws_bytes, void* stream);

/* moe_dispatch_align implements the drop policy only: with
 * cfg->overflow_policy == MOE_OVERFLOW_REROUTE and a capacity in force, or with
 * expert-choice routing, it returns MOE_ERR_INVALID_ARG rather than dropping
 * routes the caller asked to keep (use the two entry points below). */

/* Capacity dispatch with the reroute overflow policy, then the same stable
 * alignment.  Phase one is moe_dispatch_align's capacity rule.  Phase two
 * takes the routes it would drop in ascending route id; each goes to the
 * best-ranked expert of its token (the router's order on logits [T, N], the
 * fp32 logits of every expert, e.g. from moe_router_logits) that has room left
 * and that the token does not use yet (its k chosen experts and the targets of
 * its earlier slots).  A route with no such expert is dropped.  The rerouted
 * route keeps its slot j and gate; moe_combine needs nothing else.
 * Outputs as moe_dispatch_align, plus
 *   route_expert [T*k] int32, expert each route is sent to, -1 if dropped
 *   num_rerouted [1] int32;  num_dropped counts the routes left dropped;
 *   expert_counts counts all routes each expert processes.
 * Integer results only: identical bits on every run.  cfg->overflow_policy is
 * not consulted (this entry point is the reroute policy). */
moe_status moe_dispatch_align_reroute(const moe_config* cfg, int32_t T, const int32_t* topk_idx,
                                      const float* logits, uint8_t* route_kept, int32_t* route_expert,
                                      int32_t* route_pos, int32_t* sorted_route_ids,
                                      int32_t* block_expert, int32_t* num_padded,
                                      int32_t* expert_counts, int32_t* num_dropped,
                                      int32_t* num_rerouted, void* ws, size_t ws_bytes, void* stream);

/* Expert-choice routing with its padded layout (cfg->routing must be
 * MOE_ROUTING_EXPERT_CHOICE).  From logits [T, N] (moe_router_logits) every
 * expert takes its C = moe_capacity(cfg, T) tokens of largest probability:
 * the key is log p = (l - m) - log(sum_e exp(l_e - m)) in fp64 (m = largest
 * logit, sum in ascending e; NaN logits rank last), equal keys by lower token
 * index.  A token may be taken by no expert (its output is then h plus the
 * shared expert).  Routes are r = t*N + e:
 *   gates       [T*N] fp32 out, softmax probability of every (t, e)
 *   route_kept  [T*N] uint8 out, 1 if expert e took token t
 *   route_pos   [T*N] int32 out, row in sorted_route_ids, -1 if not taken
 *   sorted_route_ids [moe_max_padded_rows], block_expert [moe_max_blocks],
 *   num_padded [1], expert_counts [N] (= C for every expert): as in
 *   moe_dispatch_align, expert e's tokens in ascending t, padded with T*N.
 * moe_expert_ffn and moe_combine then run with N slots per token. */
moe_status moe_route_expert_choice(const moe_config* cfg, int32_t T, const float* logits,
                                   float* gates, uint8_t* route_kept, int32_t* route_pos,
                                   int32_t* sorted_route_ids, int32_t* block_expert,
                                   int32_t* num_padded, int32_t* expert_counts, void* ws,
                                   size_t ws_bytes, void* stream);

/* The routing_stats probe of "Mixture-of-Experts Routing at Inference Time"
 * (section "The hard part: token dropping is a silent correctness bug") on
 * topk_idx [T, k] (token choice): expert_load [N] int32 out (routes naming
 * each expert), stats (device) out.  capacity_factor sets the probe's own
 * capacity floor(mean * cf) (1.25 in the page's probe); it is independent of
 * the layer's capacity.  fp64 results are single IEEE operations on the
 * integer counts.  Asynchronous; ids outside [0, N) are not counted. */
moe_status moe_routing_stats(const moe_config* cfg, int32_t T, const int32_t* topk_idx,
                             double capacity_factor, int32_t* expert_load, moe_route_stats* stats,
                             void* stream);

/* Router margin per token ("Mixture-of-experts routing and LLM
 * repeatability"): margin [T] fp64 out = l_(k) - l_(k+1), the k-th and
 * (k+1)-th logits of logits [T, N] under the router's ranking, as the fp64
 * difference of the two fp32 values; +inf when k = N, NaN if either is NaN.
 * A small margin marks a token whose experts a small numerical change can
 * flip. */
moe_status moe_router_margin(const moe_config* cfg, int32_t T, const float* logits, double* margin,
                             void* stream);

/* Grouped SwiGLU expert FFN over the padded blocks, on tcgen05 tensor cores:
 *   for every padded row p of expert e = block_expert[p / B] with route r:
 *     x = h[r / S] (S = k, or N for expert choice; zero for the sentinel),
 *     [g | u] = x . W13_e,
 *     a = bf16(silu(g) * u), y_perm[p] = bf16(a . W2_e)  (fp32 accumulation)
 *   and, when cfg->shared_intermediate > 0, y_shared[t] = SwiGLU_shared(h[t]).
 *   w13 [N, H, 2I] bf16 (gate columns 0..I-1, up columns I..2I-1),
 *   w2 [N, I, H] bf16, w13_shared [H, 2Is], w2_shared [Is, H] (or NULL when
 *   Is == 0); y_perm [moe_max_padded_rows, H] bf16 out; y_shared [T, H] bf16
 *   out or NULL when Is == 0 (the expert outputs are stored in bf16: half the
 *   bytes of the W2 store and of the combine's reads; every sum stays fp32).
 *   Rows of y_perm that hold the sentinel, and rows past *num_padded, are
 *   not written.
 * One tile shape and one K order for every T, no split-K: each y row
 * depends only on its own x row and the expert's weights. */
moe_status moe_expert_ffn(const moe_config* cfg, int32_t T, const uint16_t* h, const uint16_t* w13,
                          const uint16_t* w2, const uint16_t* w13_shared,
                          const uint16_t* w2_shared, const int32_t* sorted_route_ids,
                          const int32_t* block_expert, const int32_t* num_padded, uint16_t* y_perm,
                          uint16_t* y_shared, void* ws, size_t ws_bytes, void* stream);

/* Gate-weighted combine into the residual:
 *   out[t] = bf16( h[t] + sum_{j ascending, kept} topk_gate[t,j] * y_perm[route_pos[t*S+j]]
 *                  + y_shared[t] )
 * accumulated in fp32 in that fixed order (y_perm, y_shared bf16 as written
 * by moe_expert_ffn); S = k slots per token (N for expert choice, whose
 * gates are the [T, N] probabilities).  y_shared may be NULL.  out [T,H]
 * bf16. */
moe_status moe_combine(const moe_config* cfg, int32_t T, const uint16_t* h, const float* topk_gate,
                       const uint8_t* route_kept, const int32_t* route_pos, const uint16_t* y_perm,
                       const uint16_t* y_shared, uint16_t* out, void* stream);

/* The whole layer: moe_route -> moe_dispatch_align -> moe_expert_ffn ->
 * moe_combine on `stream`, intermediates in the workspace.  No host
 * synchronisation and no device-to-host copy.  With the reroute policy (and
 * a capacity) the router computes every logit canonically and the dispatch is
 * moe_dispatch_align_reroute; with expert-choice routing it is
 * moe_router_logits -> moe_route_expert_choice -> moe_expert_ffn ->
 * moe_combine. */
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

/* Number of kernel launches one moe_forward of T tokens makes for this
 * configuration (the router takes two on CUDA cores or six on the tensor
 * cores; at most 1024 routes are dispatched and cut into both GEMM tile lists
 * in one launch; for at most two tokens the router's chunk sums are followed
 * by one launch that routes, dispatches and gathers the routed rows, so a
 * forward without a shared expert is five launches). */
int32_t moe_forward_launch_count(const moe_config* cfg, int32_t T);

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
 *     before any stream capture.  A new context on the device (after
 *     cudaDeviceReset, for example) moves the array: the next call notices
 *     the change of context and looks the address up again, so make the
 *     first call after a reset before any capture too.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents (the call clears what must start at zero).  Calls that
 *     overlap on the GPU (e.g. on two streams at once) race on it: order them. */
moe_status moe_dispatch_align_noalloc(const moe_config* cfg, int32_t T, const int32_t* topk_idx,
                                      uint8_t* route_kept, int32_t* route_pos,
                                      int32_t* sorted_route_ids, int32_t* block_expert,
                                      int32_t* num_padded, int32_t* expert_counts,
                                      int32_t* num_dropped, int32_t* status_out, void* stream);

/* Reads the device status word of `ws` (synchronises `stream`): the whole word
 * in *status_out; MOE_ERR_DEVICE if any bit of MOE_DEV_ERR_MASK is set. */
moe_status moe_get_device_status(const void* ws, int32_t* status_out, void* stream);

/* Clears the device status word of `ws` (asynchronous on `stream`). */
moe_status moe_clear_device_status(void* ws, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_API_H */
