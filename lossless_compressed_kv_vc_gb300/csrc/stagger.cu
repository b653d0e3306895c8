// Planner of the two alternating groups of cross-resource staggering (host code only).
//
// "VeriCache: Turning Lossy KV Cache into Lossless LLM Inference", "Cross-resource staggering
// (P1)": drafting is bound by HBM bandwidth and verification of an offloaded request by the host
// link, so some requests draft while the KV_full of others is copied in and verified. The period
// model and the exact split are stated in include/vc.h (vc_plan_stagger).
#include "vc.h"

#include <cstdint>

namespace {

constexpr int64_t kMaxCost = int64_t(1) << 40;

inline int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

bool costs_ok(const vc_stagger_cost* c, int32_t n) {
  for (int32_t r = 0; r < n; ++r)
    if (c[r].draft_ns < 0 || c[r].verify_ns < 0 || c[r].stage_ns < 0 || c[r].draft_ns > kMaxCost ||
        c[r].verify_ns > kMaxCost || c[r].stage_ns > kMaxCost)
      return false;
  return true;
}

// Twice the steady-state period of split (A, B): the largest cycle mean of the schedule's
// dependency graph, doubled so that the two-period cycles stay integers.
//   compute: draft A -> verify B -> draft B -> verify A -> (next period);  copy: copy B -> copy A
//   verify X after copy X; copy X after the previous verify X.
// Cycles (weight / periods spanned): the compute loop (D + V) / 1, the copy loop S / 1, copy X then
// verify X (S_X + V_X) / 1, and the two loops through both streams (S + V + D_X) / 2.
inline int64_t period2(int64_t dA, int64_t sA, int64_t vA, int64_t D, int64_t S, int64_t V) {
  int64_t t = 2 * (D + V);
  t = max64(t, 2 * S);
  t = max64(t, 2 * (sA + vA));
  t = max64(t, 2 * ((S - sA) + (V - vA)));
  t = max64(t, S + V + dA);
  t = max64(t, S + V + (D - dA));
  return t;
}

}  // namespace

extern "C" vc_status vc_stagger_period(const vc_stagger_cost* cost, int32_t n, const int32_t* group,
                                       int64_t* period_ns) {
  if (!cost || !group || !period_ns || n < 1) return VC_ERR_INVALID;
  if (!costs_ok(cost, n)) return VC_ERR_INVALID;
  int64_t D = 0, S = 0, V = 0, dA = 0, sA = 0, vA = 0;
  for (int32_t r = 0; r < n; ++r) {
    if (group[r] != 0 && group[r] != 1) return VC_ERR_INVALID;
    D += cost[r].draft_ns;
    S += cost[r].stage_ns;
    V += cost[r].verify_ns;
    if (group[r] == 0) {
      dA += cost[r].draft_ns;
      sA += cost[r].stage_ns;
      vA += cost[r].verify_ns;
    }
  }
  *period_ns = (period2(dA, sA, vA, D, S, V) + 1) / 2;
  return VC_OK;
}

extern "C" vc_status vc_plan_stagger(const vc_stagger_cost* cost, int32_t n, int32_t* group, int64_t* period_ns) {
  if (!cost || !group || n < 1) return VC_ERR_INVALID;
  if (n > VC_STAGGER_MAX) return VC_ERR_UNSUPPORTED;
  if (!costs_ok(cost, n)) return VC_ERR_INVALID;
  int64_t D = 0, S = 0, V = 0;
  for (int32_t r = 0; r < n; ++r) {
    D += cost[r].draft_ns;
    S += cost[r].stage_ns;
    V += cost[r].verify_ns;
  }
  // bit r-1 of the mask = group of request r (request 0 stays in A); start with everyone in A and
  // walk the reflected Gray code, which flips one request per step. Mask 0 (B empty) is a split
  // only when there is a single request.
  const uint32_t count = 1u << (n - 1);
  uint32_t mask = 0, best_mask = 0;
  int64_t dA = D, sA = S, vA = V;
  int64_t best = n == 1 ? period2(dA, sA, vA, D, S, V) : INT64_MAX;
  for (uint32_t i = 1; i < count; ++i) {
    const int bit = __builtin_ctz(i);
    const vc_stagger_cost& c = cost[bit + 1];
    mask ^= 1u << bit;
    if (mask & (1u << bit)) {  // request bit+1 moved to B
      dA -= c.draft_ns;
      sA -= c.stage_ns;
      vA -= c.verify_ns;
    } else {
      dA += c.draft_ns;
      sA += c.stage_ns;
      vA += c.verify_ns;
    }
    const int64_t t = period2(dA, sA, vA, D, S, V);
    if (t < best || (t == best && mask < best_mask)) {
      best = t;
      best_mask = mask;
    }
  }
  group[0] = 0;
  for (int32_t r = 1; r < n; ++r) group[r] = (int32_t)((best_mask >> (r - 1)) & 1u);
  if (period_ns) *period_ns = (best + 1) / 2;
  return VC_OK;
}
