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
 * (no shared expert).  out [T,H] bf16 bits. */
void oracle_moe_forward(int32_t T, int32_t H, int32_t N, int32_t k, int32_t I, int32_t B,
                        double capacity_factor, int32_t Is, const uint16_t* h,
                        const uint16_t* w_gate, const float* bias, const uint16_t* w13,
                        const uint16_t* w2, const uint16_t* w13s, const uint16_t* w2s,
                        uint16_t* out, int32_t nthreads);

/* Round a double to the nearest bf16 (ties to even); returns the bit pattern. */
uint16_t oracle_bf16_round(double x);

#ifdef __cplusplus
}
#endif
#endif
