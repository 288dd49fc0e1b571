/*
 * CPU oracle for the batch-invariant Mixture-of-Experts layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, scalar C++ restatement of
 * what the layer computes, written from the method's published description.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load it.  It shares no code with the CUDA path.
 *
 * Conventions: all arrays are host memory, row-major; bf16 values are passed
 * as their uint16 bit patterns; routes are numbered r = t*k + j (token t,
 * slot j), the flattened route identifier of "Route-Block Membership Selects
 * Packed-AWQ Arithmetic" (section "The bookkeeping before the matrix
 * multiplication").
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

/* Router projection l = h . W_g (+ bias), fp32, in the fixed chunked order:
 * the hidden dimension is cut into 256-element chunks; each chunk is summed
 * sequentially from +0 in ascending index; the chunk sums are added
 * sequentially, in ascending chunk order, to a total that starts at +0; the
 * bias (if any) is added last.  h [T,H], w_gate [H,N], bias [N] or NULL,
 * logits [T,N]. */
void oracle_router_logits(int32_t T, int32_t H, int32_t N, const uint16_t* h,
                          const uint16_t* w_gate, const float* bias, float* logits,
                          int32_t nthreads);

/* Top-k under the total order (larger logit first; equal logits: lower expert
 * index first; NaN below every number), slots stored by ascending expert
 * index.  Gates are the softmax renormalised over the selected experts,
 * computed in fp64.  topk_idx [T,k], gates [T,k]. */
void oracle_select_topk(int32_t T, int32_t N, int32_t k, const float* logits,
                        int32_t* topk_idx, double* gates);

/* Router margin l_(k) - l_(k+1) per token (fp64 of the fp32 logits; +inf if k == N). */
void oracle_router_margin(int32_t T, int32_t N, int32_t k, const float* logits, double* margin);

/* Expert capacity ceil(cf*T*k/N) for cf > 0, else -1 (no limit). */
int32_t oracle_capacity(int32_t T, int32_t N, int32_t k, double capacity_factor);

/* Capacity-limited dispatch and stable alignment into padded blocks.
 * capacity < 0 means no limit.  Outputs:
 *   route_kept [R]        1 if the route was kept, else 0
 *   route_pos [R]         row of the route in sorted_route_ids, -1 if dropped
 *   sorted_route_ids [*]  per expert e = 0..N-1: its kept routes in ascending
 *                         r, padded with the sentinel R up to a multiple of B
 *   block_expert [*]      expert of each B-row block
 *   num_padded [1], expert_counts [N] (kept), num_dropped [1]
 * Entries of topk_idx outside [0,N) are treated as not routed (kept = 0). */
void oracle_dispatch(int32_t T, int32_t N, int32_t k, int32_t B, int32_t capacity,
                     const int32_t* topk_idx, uint8_t* route_kept, int32_t* route_pos,
                     int32_t* sorted_route_ids, int32_t* block_expert, int32_t* num_padded,
                     int32_t* expert_counts, int32_t* num_dropped);

/* Overflow policy "reroute" ("Mixture-of-Experts Routing at Inference Time",
 * Figure 2 and the mitigations after routing_stats: an overflowing token goes
 * to its next-choice expert instead of skipping the expert tier).
 * Phase 1 is the drop policy's capacity rule (each expert keeps its first
 * `capacity` routes by ascending route id).  Phase 2 takes the routes that
 * overflowed, in ascending route id; each goes to the best-ranked expert (the
 * top-k total order on the token's logits) that still has room and that the
 * token does not already use (its k chosen experts and the targets of its
 * earlier slots).  A route with no such expert stays dropped.
 *   route_expert [R]  expert the route is finally sent to, -1 if dropped
 * capacity < 0 (no limit): nothing overflows.  Entries of topk_idx outside
 * [0, N) are not routed (-1, not counted). */
void oracle_reroute(int32_t T, int32_t N, int32_t k, int32_t capacity, const float* logits,
                    const int32_t* topk_idx, int32_t* route_expert, int32_t* num_rerouted,
                    int32_t* num_dropped);

/* routing_stats of "Mixture-of-Experts Routing at Inference Time" (section
 * "The hard part"): per-expert load = number of routes in topk_idx [T, k]
 * naming the expert (ids outside [0, N) are ignored); mean = total / N;
 * probe capacity = floor(mean * capacity_factor); dropped = sum over experts
 * of max(0, load - capacity).  All in fp64:
 *   load [N];  ints = {max_load, min_load, capacity, dropped, total}
 *   reals = {imbalance_ratio = max_load / mean, drop_fraction = dropped / total}
 * With no routes every output is 0. */
void oracle_routing_stats(int32_t T, int32_t N, int32_t k, const int32_t* topk_idx,
                          double capacity_factor, int32_t* load, int32_t* ints, double* reals);

/* Expert-choice routing ("Mixture-of-experts routing and LLM repeatability":
 * each expert takes its highest-scoring tokens of the batch; "Mixture-of-
 * Experts Routing at Inference Time", section "Integration: where routing
 * lives in a serving stack", the comparison of routing variants: each expert
 * picks the tokens it will take, up to its capacity).  Scores are the softmax
 * probabilities over the N experts.  Routes are r = t*N + e.
 *   key[t,e] = (l[t,e] - m) - log(sum_e exp(l[t,e] - m))   (fp64, the log
 *              of the probability; m = max non-NaN logit, the sum in
 *              ascending e, NaN logits left out of it and given a NaN key)
 *   expert e takes the `capacity` tokens with the largest key (NaN lowest,
 *   equal keys: lower token index first); capacity is clipped to T.
 *   selected [T*N] 1 if expert e took token t;  probs [T*N] = exp(key). */
void oracle_expert_choice(int32_t T, int32_t N, int32_t capacity, const float* logits,
                          uint8_t* selected, double* probs);

/* Capacity of expert-choice routing: ceil(cf*T*k/N) with cf = 1 when cf <= 0,
 * clipped to T. */
int32_t oracle_ec_capacity(int32_t T, int32_t N, int32_t k, double capacity_factor);

/* SwiGLU expert on one token row, fp64 accumulation:
 *   g = x . W13[:, 0:I], u = x . W13[:, I:2I], a = bf16(silu(g) * u), y = a . W2
 * x [H] bf16, w13 [H, 2I], w2 [I, H]; y [H] fp64; a_out [I] bf16 bits or NULL. */
void oracle_expert_row(int32_t H, int32_t I, const uint16_t* x, const uint16_t* w13,
                       const uint16_t* w2, double* y, uint16_t* a_out);

/* The expert outputs of a list of routes, in parallel over routes.
 * tokens[n], experts[n] select x = h[tokens[i]] and the expert's weights in
 * w13 [N,H,2I], w2 [N,I,H]; y [n,H] fp64. */
void oracle_expert_rows(int32_t n, const int32_t* tokens, const int32_t* experts, int32_t H,
                        int32_t I, const uint16_t* h, const uint16_t* w13, const uint16_t* w2,
                        double* y, int32_t nthreads);

/* Gate-weighted combine into the residual for a list of tokens:
 *   out[t] = bf16( h[t] + sum over kept slots j (ascending) gates[t,j]*y_route[t,j] + y_shared[t] )
 * y_route [n, k, H] fp64 (only kept slots are read), y_shared [n, H] fp64 or
 * NULL; out [n, H] bf16 bits. */
void oracle_combine_rows(int32_t n, const int32_t* tokens, int32_t H, int32_t k,
                         const uint16_t* h, const double* gates, const uint8_t* route_kept,
                         const double* y_route, const double* y_shared, uint16_t* out);

/* Whole layer for all T tokens (small shapes): router, top-k, capacity,
 * alignment, routed and shared SwiGLU experts, combine.  w13s/w2s may be NULL
 * (no shared expert).  overflow_policy 0 drops overflowing routes, 1 reroutes
 * them (oracle_reroute; the route keeps its slot's gate).  routing 0 is
 * token choice (top-k), 1 is expert choice (oracle_expert_choice; a token's
 * routes are its N slots e = 0..N-1, gate = probability, summed in ascending
 * e).  out [T,H] bf16 bits. */
void oracle_moe_forward(int32_t T, int32_t H, int32_t N, int32_t k, int32_t I, int32_t B,
                        double capacity_factor, int32_t overflow_policy, int32_t routing,
                        int32_t Is, const uint16_t* h,
                        const uint16_t* w_gate, const float* bias, const uint16_t* w13,
                        const uint16_t* w2, const uint16_t* w13s, const uint16_t* w2s,
                        uint16_t* out, int32_t nthreads);

/* Round a double to the nearest bf16 (ties to even); returns the bit pattern. */
uint16_t oracle_bf16_round(double x);

#ifdef __cplusplus
}
#endif
#endif
