// CPU oracle for the batch-invariant MoE layer forward.
//
// TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
// benchmark's CPU-baseline leg, never by the product path.  Plain scalar
// C++17, compiled -O2 -ffp-contract=off without fast-math.  Every function
// follows one passage of the pages that define the method:
//
//  * "Mixture-of-Experts Routing at Inference Time" (ACE Journal), section
//    "How sparse routing works" and its TopKRouter: one router matrix W_g
//    [hidden, N] maps a token to N logits; softmax, keep the k best, rescale
//    their gates to sum to one; the token's result adds each kept expert's
//    output weighted by its gate.
//  * Same page, "The hard part: token dropping is a silent correctness bug"
//    and Figure 2: a route that overflows its expert's capacity contributes
//    nothing; the token keeps its residual plus its other kept routes.
//  * "Mixture-of-experts routing and LLM repeatability"
//    (vincentschmalbach.com): the per-token pseudo-code (scores, top_k,
//    gate-weighted sum into the residual stream), the Switch capacity rule
//    (tokens/experts x capacity factor) and in-order filling of capacity.
//  * "Why temperature=0 Still Gives Different Answers: Batch Invariance",
//    Tier 2 of "How do I make LLM inference reproducible?": a reduction cut
//    into constant 256-element pieces added in one order (the router's fp32
//    summation order below).
//  * "Route-Block Membership Selects Packed-AWQ Arithmetic", sections "The
//    bookkeeping before the matrix multiplication" and "Stable construction
//    selected a third trajectory": routed rows are grouped per expert and
//    padded to whole blocks; the kept routes are sorted by expert id, then by
//    flattened route id.
#include "moe_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

double silu(double g) { return g / (1.0 + std::exp(-g)); }

// Runs body(i) for i in [0, n) on up to nthreads std::threads, contiguous
// ranges per thread.  Every i is computed by exactly one thread in the same
// way, so results do not depend on the thread count.
template <class F>
void parallel_for(int64_t n, int32_t nthreads, F body) {
  if (nthreads <= 0) nthreads = (int32_t)std::max(1u, std::thread::hardware_concurrency());
  if (n <= 1 || nthreads == 1) {
    for (int64_t i = 0; i < n; ++i) body(i);
    return;
  }
  int64_t nt = std::min<int64_t>(nthreads, n);
  int64_t per = (n + nt - 1) / nt;
  std::vector<std::thread> pool;
  for (int64_t t = 0; t < nt; ++t) {
    int64_t b = t * per, e = std::min(n, b + per);
    if (b >= e) break;
    pool.emplace_back([=, &body] {
      for (int64_t i = b; i < e; ++i) body(i);
    });
  }
  for (auto& th : pool) th.join();
}

// Ranking of two experts for top-k: true if (la, a) comes before (lb, b).
bool ranks_before(float la, int32_t a, float lb, int32_t b) {
  bool na = std::isnan(la), nb = std::isnan(lb);
  if (na != nb) return nb;           // a number ranks above NaN
  if (!na && la != lb) return la > lb;
  return a < b;                      // equal scores (or both NaN): lower index first
}

}  // namespace

extern "C" {

uint16_t oracle_bf16_round(double x) {
  // Nearest bf16 to x, ties to even: bf16 keeps 8 significant bits and the
  // fp32 exponent range.
  if (std::isnan(x)) return 0x7FC0;
  if (x == 0.0) return std::signbit(x) ? 0x8000 : 0x0000;
  if (std::isinf(x)) return std::signbit(x) ? 0xFF80 : 0x7F80;
  int e = 0;
  std::frexp(x, &e);                       // |x| = m * 2^e, 0.5 <= m < 1
  int ulp_exp = std::max(e - 8, -133);     // bf16 subnormal spacing is 2^-133
  double q = std::ldexp(x, -ulp_exp);      // exact scaling
  double r = std::nearbyint(q);            // default rounding: nearest, ties to even
  double v = std::ldexp(r, ulp_exp);
  float f = (float)v;                      // exactly representable in fp32 (or overflows to inf)
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

void oracle_router_logits(int32_t T, int32_t H, int32_t N, const uint16_t* h,
                          const uint16_t* w_gate, const float* bias, float* logits,
                          int32_t nthreads) {
  const int32_t chunk = 256;
  parallel_for(T, nthreads, [&](int64_t t) {
    const uint16_t* x = h + (size_t)t * H;
    for (int32_t e = 0; e < N; ++e) {
      float total = 0.0f;
      for (int32_t c0 = 0; c0 < H; c0 += chunk) {
        float part = 0.0f;
        int32_t c1 = std::min(H, c0 + chunk);
        for (int32_t i = c0; i < c1; ++i) {
          float prod = bf16_to_float(x[i]) * bf16_to_float(w_gate[(size_t)i * N + e]);  // exact in fp32
          part = part + prod;
        }
        total = total + part;
      }
      if (bias) total = total + bias[e];
      logits[(size_t)t * N + e] = total;
    }
  });
}

void oracle_select_topk(int32_t T, int32_t N, int32_t k, const float* logits,
                        int32_t* topk_idx, double* gates) {
  std::vector<int32_t> order(N);
  for (int32_t t = 0; t < T; ++t) {
    const float* l = logits + (size_t)t * N;
    for (int32_t e = 0; e < N; ++e) order[e] = e;
    std::sort(order.begin(), order.end(),
              [&](int32_t a, int32_t b) { return ranks_before(l[a], a, l[b], b); });
    std::vector<int32_t> sel(order.begin(), order.begin() + k);
    std::sort(sel.begin(), sel.end());   // slots by ascending expert index
    // softmax over all N then renormalising over the selected k equals the
    // softmax over the selected logits alone (the full denominator cancels)
    double m = -std::numeric_limits<double>::infinity();
    for (int32_t j = 0; j < k; ++j) m = std::max(m, (double)l[sel[j]]);
    double s = 0.0;
    std::vector<double> ex(k);
    for (int32_t j = 0; j < k; ++j) {
      ex[j] = std::exp((double)l[sel[j]] - m);
      s += ex[j];
    }
    for (int32_t j = 0; j < k; ++j) {
      topk_idx[(size_t)t * k + j] = sel[j];
      gates[(size_t)t * k + j] = ex[j] / s;
    }
  }
}

void oracle_router_margin(int32_t T, int32_t N, int32_t k, const float* logits, double* margin) {
  std::vector<int32_t> order(N);
  for (int32_t t = 0; t < T; ++t) {
    const float* l = logits + (size_t)t * N;
    if (k >= N) {
      margin[t] = std::numeric_limits<double>::infinity();
      continue;
    }
    for (int32_t e = 0; e < N; ++e) order[e] = e;
    std::sort(order.begin(), order.end(),
              [&](int32_t a, int32_t b) { return ranks_before(l[a], a, l[b], b); });
    margin[t] = (double)l[order[k - 1]] - (double)l[order[k]];
  }
}

int32_t oracle_capacity(int32_t T, int32_t N, int32_t k, double capacity_factor) {
  if (!(capacity_factor > 0.0)) return -1;
  return (int32_t)std::ceil(capacity_factor * (double)T * (double)k / (double)N);
}

void oracle_dispatch(int32_t T, int32_t N, int32_t k, int32_t B, int32_t capacity,
                     const int32_t* topk_idx, uint8_t* route_kept, int32_t* route_pos,
                     int32_t* sorted_route_ids, int32_t* block_expert, int32_t* num_padded,
                     int32_t* expert_counts, int32_t* num_dropped) {
  const int64_t R = (int64_t)T * k;
  const int32_t sentinel = (int32_t)R;
  // Capacity is filled in batch order: an expert's routes are taken by
  // ascending route id (= ascending token index) and the first `capacity`
  // are kept.
  std::vector<std::vector<int32_t>> kept(N);
  std::vector<int64_t> load(N, 0);
  for (int64_t r = 0; r < R; ++r) {
    int32_t e = topk_idx[r];
    route_kept[r] = 0;
    route_pos[r] = -1;
    if (e < 0 || e >= N) continue;
    if (capacity < 0 || load[e] < capacity) {
      kept[e].push_back((int32_t)r);
      route_kept[r] = 1;
    }
    load[e] += 1;
  }
  // Stable construction: segments in ascending expert id, each segment's
  // routes in ascending route id, padded with the sentinel to a multiple of B.
  int64_t row = 0, block = 0, dropped = 0;
  for (int32_t e = 0; e < N; ++e) {
    int64_t cnt = (int64_t)kept[e].size();
    int64_t padded = (cnt + B - 1) / B * B;
    for (int64_t j = 0; j < cnt; ++j) {
      sorted_route_ids[row + j] = kept[e][j];
      route_pos[kept[e][j]] = (int32_t)(row + j);
    }
    for (int64_t j = cnt; j < padded; ++j) sorted_route_ids[row + j] = sentinel;
    for (int64_t b = 0; b < padded / B; ++b) block_expert[block + b] = e;
    row += padded;
    block += padded / B;
    expert_counts[e] = (int32_t)cnt;
    dropped += load[e] - cnt;
  }
  *num_padded = (int32_t)row;
  *num_dropped = (int32_t)dropped;
}

void oracle_reroute(int32_t T, int32_t N, int32_t k, int32_t capacity, const float* logits,
                    const int32_t* topk_idx, int32_t* route_expert, int32_t* num_rerouted,
                    int32_t* num_dropped) {
  const int64_t R = (int64_t)T * k;
  std::vector<int64_t> used(N, 0);
  // phase 1: the drop policy's rule, first `capacity` routes of each expert
  for (int64_t r = 0; r < R; ++r) {
    int32_t e = topk_idx[r];
    route_expert[r] = -1;
    if (e < 0 || e >= N) continue;
    if (capacity < 0 || used[e] < capacity) {
      route_expert[r] = e;
      used[e] += 1;
    }
  }
  int32_t rerouted = 0, dropped = 0;
  // phase 2: overflowing routes in ascending route id, each to the token's
  // best-ranked expert with room that the token does not use yet
  std::vector<int32_t> order(N);
  for (int64_t r = 0; r < R && capacity >= 0; ++r) {
    int32_t e = topk_idx[r];
    if (e < 0 || e >= N || route_expert[r] >= 0) continue;
    const int64_t t = r / k;
    const float* l = logits + (size_t)t * N;
    for (int32_t x = 0; x < N; ++x) order[x] = x;
    std::sort(order.begin(), order.end(),
              [&](int32_t a, int32_t b) { return ranks_before(l[a], a, l[b], b); });
    int32_t target = -1;
    for (int32_t cand : order) {
      if (used[cand] >= capacity) continue;
      bool taken = false;
      for (int64_t q = t * k; q < (t + 1) * k; ++q)
        if (topk_idx[q] == cand || (q < r && route_expert[q] == cand)) taken = true;
      if (taken) continue;
      target = cand;
      break;
    }
    if (target >= 0) {
      route_expert[r] = target;
      used[target] += 1;
      ++rerouted;
    } else {
      ++dropped;
    }
  }
  *num_rerouted = rerouted;
  *num_dropped = dropped;
}

void oracle_routing_stats(int32_t T, int32_t N, int32_t k, const int32_t* topk_idx,
                          double capacity_factor, int32_t* load, int32_t* ints, double* reals) {
  for (int32_t e = 0; e < N; ++e) load[e] = 0;
  int64_t total = 0;
  for (int64_t r = 0; r < (int64_t)T * k; ++r) {
    int32_t e = topk_idx[r];
    if (e < 0 || e >= N) continue;
    load[e] += 1;
    total += 1;
  }
  for (int i = 0; i < 5; ++i) ints[i] = 0;
  reals[0] = reals[1] = 0.0;
  if (total == 0) return;
  int32_t mx = load[0], mn = load[0];
  for (int32_t e = 1; e < N; ++e) {
    mx = std::max(mx, load[e]);
    mn = std::min(mn, load[e]);
  }
  const double mean = (double)total / (double)N;
  const int32_t cap = (int32_t)std::floor(mean * capacity_factor);
  int64_t drops = 0;
  for (int32_t e = 0; e < N; ++e) drops += std::max<int64_t>(0, (int64_t)load[e] - cap);
  ints[0] = mx;
  ints[1] = mn;
  ints[2] = cap;
  ints[3] = (int32_t)drops;
  ints[4] = (int32_t)total;
  reals[0] = (double)mx / mean;
  reals[1] = (double)drops / (double)total;
}

int32_t oracle_ec_capacity(int32_t T, int32_t N, int32_t k, double capacity_factor) {
  const double cf = capacity_factor > 0.0 ? capacity_factor : 1.0;
  const int32_t c = (int32_t)std::ceil(cf * (double)T * (double)k / (double)N);
  return std::min(c, T);
}

void oracle_expert_choice(int32_t T, int32_t N, int32_t capacity, const float* logits,
                          uint8_t* selected, double* probs) {
  std::vector<double> key((size_t)T * N);
  for (int32_t t = 0; t < T; ++t) {
    const float* l = logits + (size_t)t * N;
    double m = -std::numeric_limits<double>::infinity();
    for (int32_t e = 0; e < N; ++e)
      if (!std::isnan(l[e])) m = std::max(m, (double)l[e]);
    double s = 0.0;
    for (int32_t e = 0; e < N; ++e)
      if (!std::isnan(l[e])) s += std::exp((double)l[e] - m);
    const double log_s = std::log(s);
    for (int32_t e = 0; e < N; ++e) {
      // log p = (l - m) - log(sum): shifting all of a token's logits by a
      // constant leaves every term, and so the key, unchanged
      const double kv = std::isnan(l[e]) ? std::numeric_limits<double>::quiet_NaN()
                                         : ((double)l[e] - m) - log_s;
      key[(size_t)t * N + e] = kv;
      probs[(size_t)t * N + e] = std::exp(kv);
      selected[(size_t)t * N + e] = 0;
    }
  }
  const int32_t C = std::min(std::max(capacity, 0), T);
  std::vector<int32_t> order(T);
  for (int32_t e = 0; e < N; ++e) {
    for (int32_t t = 0; t < T; ++t) order[t] = t;
    // larger key first, NaN last, equal keys by lower token index
    std::sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
      const double ka = key[(size_t)a * N + e], kb = key[(size_t)b * N + e];
      const bool na = std::isnan(ka), nb = std::isnan(kb);
      if (na != nb) return nb;
      if (!na && ka != kb) return ka > kb;
      return a < b;
    });
    for (int32_t i = 0; i < C; ++i) selected[(size_t)order[i] * N + e] = 1;
  }
}

void oracle_expert_row(int32_t H, int32_t I, const uint16_t* x, const uint16_t* w13,
                       const uint16_t* w2, double* y, uint16_t* a_out) {
  std::vector<double> g(I, 0.0), u(I, 0.0);
  for (int32_t i = 0; i < H; ++i) {
    double xi = bf16_to_float(x[i]);
    const uint16_t* row = w13 + (size_t)i * 2 * I;
    for (int32_t n = 0; n < I; ++n) {
      g[n] += xi * bf16_to_float(row[n]);
      u[n] += xi * bf16_to_float(row[I + n]);
    }
  }
  std::vector<double> a(I);
  for (int32_t n = 0; n < I; ++n) {
    // the activation is stored in the layer's bf16 activation type
    uint16_t ab = oracle_bf16_round(silu(g[n]) * u[n]);
    if (a_out) a_out[n] = ab;
    a[n] = bf16_to_float(ab);
  }
  for (int32_t d = 0; d < H; ++d) y[d] = 0.0;
  for (int32_t n = 0; n < I; ++n) {
    const uint16_t* row = w2 + (size_t)n * H;
    for (int32_t d = 0; d < H; ++d) y[d] += a[n] * bf16_to_float(row[d]);
  }
}

void oracle_expert_rows(int32_t n, const int32_t* tokens, const int32_t* experts, int32_t H,
                        int32_t I, const uint16_t* h, const uint16_t* w13, const uint16_t* w2,
                        double* y, int32_t nthreads) {
  parallel_for(n, nthreads, [&](int64_t i) {
    int32_t t = tokens[i], e = experts[i];
    oracle_expert_row(H, I, h + (size_t)t * H, w13 + (size_t)e * H * 2 * I,
                      w2 + (size_t)e * I * H, y + (size_t)i * H, nullptr);
  });
}

void oracle_combine_rows(int32_t n, const int32_t* tokens, int32_t H, int32_t k,
                         const uint16_t* h, const double* gates, const uint8_t* route_kept,
                         const double* y_route, const double* y_shared, uint16_t* out) {
  for (int32_t i = 0; i < n; ++i) {
    int32_t t = tokens[i];
    for (int32_t d = 0; d < H; ++d) {
      double acc = 0.0;
      for (int32_t j = 0; j < k; ++j) {
        size_t r = (size_t)t * k + j;
        if (!route_kept[r]) continue;   // dropped: the expert adds nothing
        acc += gates[r] * y_route[((size_t)i * k + j) * H + d];
      }
      if (y_shared) acc += y_shared[(size_t)i * H + d];
      out[(size_t)i * H + d] = oracle_bf16_round((double)bf16_to_float(h[(size_t)t * H + d]) + acc);
    }
  }
}

void oracle_moe_forward(int32_t T, int32_t H, int32_t N, int32_t k, int32_t I, int32_t B,
                        double capacity_factor, int32_t overflow_policy, int32_t routing,
                        int32_t Is, const uint16_t* h,
                        const uint16_t* w_gate, const float* bias, const uint16_t* w13,
                        const uint16_t* w2, const uint16_t* w13s, const uint16_t* w2s,
                        uint16_t* out, int32_t nthreads) {
  if (T <= 0) return;
  std::vector<float> logits((size_t)T * N);
  oracle_router_logits(T, H, N, h, w_gate, bias, logits.data(), nthreads);
  // routes: token choice has k slots per token (its top-k experts), expert
  // choice has N (slot e = expert e, routed if the expert took the token)
  const int32_t slots = routing == 1 ? N : k;
  const int64_t R = (int64_t)T * slots;
  std::vector<int32_t> route_expert(R);
  std::vector<double> gates(R);
  if (routing == 1) {
    std::vector<uint8_t> sel(R);
    oracle_expert_choice(T, N, oracle_ec_capacity(T, N, k, capacity_factor), logits.data(),
                         sel.data(), gates.data());
    for (int64_t r = 0; r < R; ++r) route_expert[r] = sel[r] ? (int32_t)(r % N) : -1;
  } else {
    std::vector<int32_t> idx(R);
    oracle_select_topk(T, N, k, logits.data(), idx.data(), gates.data());
    int32_t cap = oracle_capacity(T, N, k, capacity_factor);
    if (overflow_policy == 1) {
      int32_t rerouted = 0, dropped = 0;
      oracle_reroute(T, N, k, cap, logits.data(), idx.data(), route_expert.data(), &rerouted,
                     &dropped);
    } else {
      // drop policy: the routes kept by the capacity rule keep their expert
      std::vector<uint8_t> kept0(R);
      std::vector<int32_t> pos0(R), sorted0(R + (int64_t)N * B), blocks0(R / B + N + 1), counts0(N);
      int32_t np0 = 0, nd0 = 0;
      oracle_dispatch(T, N, k, B, cap, idx.data(), kept0.data(), pos0.data(), sorted0.data(),
                      blocks0.data(), &np0, counts0.data(), &nd0);
      for (int64_t r = 0; r < R; ++r) route_expert[r] = kept0[r] ? idx[r] : -1;
    }
  }
  // every route that has an expert is kept; the stable layout follows
  std::vector<uint8_t> kept(R);
  std::vector<int32_t> pos(R), sorted(R + (int64_t)N * B), blocks(R / B + N + 1), counts(N);
  int32_t num_padded = 0, num_dropped = 0;
  oracle_dispatch(T, N, slots, B, -1, route_expert.data(), kept.data(), pos.data(), sorted.data(),
                  blocks.data(), &num_padded, counts.data(), &num_dropped);
  // expert outputs for every kept route, stored at [t, slot]
  std::vector<int32_t> toks, exps, slot_of;
  for (int64_t r = 0; r < R; ++r)
    if (kept[r]) {
      toks.push_back((int32_t)(r / slots));
      exps.push_back(route_expert[r]);
      slot_of.push_back((int32_t)r);
    }
  std::vector<double> y_kept(toks.size() * (size_t)H);
  oracle_expert_rows((int32_t)toks.size(), toks.data(), exps.data(), H, I, h, w13, w2,
                     y_kept.data(), nthreads);
  std::vector<double> y_route((size_t)R * H, 0.0);
  for (size_t i = 0; i < slot_of.size(); ++i)
    std::memcpy(&y_route[(size_t)slot_of[i] * H], &y_kept[i * H], sizeof(double) * H);
  std::vector<double> y_shared;
  if (Is > 0 && w13s && w2s) {
    y_shared.assign((size_t)T * H, 0.0);
    parallel_for(T, nthreads, [&](int64_t t) {
      oracle_expert_row(H, Is, h + (size_t)t * H, w13s, w2s, &y_shared[(size_t)t * H], nullptr);
    });
  }
  std::vector<int32_t> all(T);
  for (int32_t t = 0; t < T; ++t) all[t] = t;
  oracle_combine_rows(T, all.data(), H, slots, h, gates.data(), kept.data(), y_route.data(),
                      y_shared.empty() ? nullptr : y_shared.data(), out);
}

}  // extern "C"
