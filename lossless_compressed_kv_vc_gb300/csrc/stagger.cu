// Planner of the two alternating groups of cross-resource staggering (host code only).
//
// "VeriCache: Turning Lossy KV Cache into Lossless LLM Inference", "Cross-resource staggering
// (P1)": drafting is bound by HBM bandwidth and verification of an offloaded request by the host
// link, so some requests draft while the KV_full of others is copied in and verified. The period
// model and the exact split are stated in include/vc.h (vc_plan_stagger).
#include "vc.h"

#include <algorithm>
#include <cstdint>
#include <vector>

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

// Tie-break of splits with equal 2T: the longer phase's GPU work, max(D_A + V_B, D_B + V_A) (phase
// 1 drafts A and verifies B, phase 2 the reverse). The period model cannot tell such splits apart
// (it is set by a bound they share, often D + V), but a lopsided split leaves one phase with little
// drafting to cover the other group's copy and with launches of little work; measured on the
// mixed workload's quantised half at its own draft lengths, request 1 alone in B ran 3.5% slower
// than halves.
inline int64_t phase_max(int64_t dA, int64_t vA, int64_t D, int64_t V) {
  return max64(dA + (V - vA), (D - dA) + vA);
}

// (2T, phase work) compared lexicographically
inline bool better(int64_t t, int64_t ph, int64_t bt, int64_t bph) { return t < bt || (t == bt && ph < bph); }

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
  int64_t best_ph = n == 1 ? phase_max(dA, vA, D, V) : INT64_MAX;
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
    const int64_t ph = phase_max(dA, vA, D, V);
    if (better(t, ph, best, best_ph) || (t == best && ph == best_ph && mask < best_mask)) {
      best = t;
      best_ph = ph;
      best_mask = mask;
    }
  }
  group[0] = 0;
  for (int32_t r = 1; r < n; ++r) group[r] = (int32_t)((best_mask >> (r - 1)) & 1u);
  if (period_ns) *period_ns = (best + 1) / 2;
  return VC_OK;
}

namespace {

// A split with group A's sums, kept in step with its moves.
struct Split {
  std::vector<int32_t> g;  // 0 = A, 1 = B
  int64_t dA = 0, sA = 0, vA = 0;
  int32_t nA = 0;
};

void sums_of(Split& sp, const vc_stagger_cost* c, int32_t n) {
  sp.dA = sp.sA = sp.vA = 0;
  sp.nA = 0;
  for (int32_t r = 0; r < n; ++r)
    if (sp.g[r] == 0) {
      sp.dA += c[r].draft_ns;
      sp.sA += c[r].stage_ns;
      sp.vA += c[r].verify_ns;
      ++sp.nA;
    }
}

// First-improvement descent: scan the single moves (request r to the other group, both groups
// staying non-empty) in index order, then the swaps (r in A with q in B) in (r, q) order; apply the
// first that lowers (2T, phase work) and start over. Stops when none does or after max_steps
// improvements.
void descend(Split& sp, const vc_stagger_cost* c, int32_t n, int64_t D, int64_t S, int64_t V, int64_t max_steps) {
  int64_t cur = period2(sp.dA, sp.sA, sp.vA, D, S, V);
  int64_t cur_ph = phase_max(sp.dA, sp.vA, D, V);
  for (int64_t step = 0; step < max_steps; ++step) {
    bool moved = false;
    for (int32_t r = 0; r < n && !moved; ++r) {
      const bool inA = sp.g[r] == 0;
      if (inA ? sp.nA == 1 : sp.nA == n - 1) continue;
      const int64_t sg = inA ? -1 : 1;
      const int64_t t = period2(sp.dA + sg * c[r].draft_ns, sp.sA + sg * c[r].stage_ns,
                                sp.vA + sg * c[r].verify_ns, D, S, V);
      const int64_t ph = phase_max(sp.dA + sg * c[r].draft_ns, sp.vA + sg * c[r].verify_ns, D, V);
      if (better(t, ph, cur, cur_ph)) {
        sp.g[r] ^= 1;
        sp.dA += sg * c[r].draft_ns;
        sp.sA += sg * c[r].stage_ns;
        sp.vA += sg * c[r].verify_ns;
        sp.nA += inA ? -1 : 1;
        cur = t;
        cur_ph = ph;
        moved = true;
      }
    }
    for (int32_t r = 0; r < n && !moved; ++r) {
      if (sp.g[r] != 0) continue;
      for (int32_t q = 0; q < n && !moved; ++q) {
        if (sp.g[q] != 1) continue;
        const int64_t dA = sp.dA - c[r].draft_ns + c[q].draft_ns;
        const int64_t sA = sp.sA - c[r].stage_ns + c[q].stage_ns;
        const int64_t vA = sp.vA - c[r].verify_ns + c[q].verify_ns;
        const int64_t t = period2(dA, sA, vA, D, S, V);
        const int64_t ph = phase_max(dA, vA, D, V);
        if (better(t, ph, cur, cur_ph)) {
          sp.g[r] = 1;
          sp.g[q] = 0;
          sp.dA = dA;
          sp.sA = sA;
          sp.vA = vA;
          cur = t;
          cur_ph = ph;
          moved = true;
        }
      }
    }
    if (!moved) return;
  }
}

}  // namespace

extern "C" vc_status vc_plan_stagger_local(const vc_stagger_cost* cost, int32_t n, int32_t* group,
                                           int64_t* period_ns) {
  if (!cost || !group || n < 1) return VC_ERR_INVALID;
  if (n > VC_STAGGER_LOCAL_MAX) return VC_ERR_UNSUPPORTED;
  if (!costs_ok(cost, n)) return VC_ERR_INVALID;
  int64_t D = 0, S = 0, V = 0;
  for (int32_t r = 0; r < n; ++r) {
    D += cost[r].draft_ns;
    S += cost[r].stage_ns;
    V += cost[r].verify_ns;
  }
  if (n == 1) {
    group[0] = 0;
    if (period_ns) *period_ns = (period2(D, S, V, D, S, V) + 1) / 2;
    return VC_OK;
  }
  // seeds: first half / second half, alternating, and a greedy pass that takes the requests by
  // decreasing d + s + v and puts each where the split-dependent part of 2T over the partial sums,
  // max(2 (S_A + V_A), 2 (S_B + V_B), S + V + D_A, S + V + D_B), comes out lower (ties: the group
  // with fewer requests, then A)
  std::vector<Split> seeds(3);
  for (auto& sp : seeds) sp.g.assign(n, 0);
  for (int32_t r = 0; r < n; ++r) {
    seeds[0].g[r] = r < (n + 1) / 2 ? 0 : 1;
    seeds[1].g[r] = r & 1;
  }
  {
    std::vector<int32_t> order(n);
    for (int32_t r = 0; r < n; ++r) order[r] = r;
    auto load = [&](int32_t r) { return cost[r].draft_ns + cost[r].stage_ns + cost[r].verify_ns; };
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return load(a) > load(b); });
    const int64_t W = S + V;
    int64_t x[2] = {0, 0}, y[2] = {0, 0};
    int32_t cnt[2] = {0, 0};
    for (int32_t r : order) {
      const int64_t xr = cost[r].stage_ns + cost[r].verify_ns, yr = cost[r].draft_ns;
      int64_t part[2];
      for (int k = 0; k < 2; ++k) {
        const int64_t x0 = x[0] + (k == 0 ? xr : 0), x1 = x[1] + (k == 1 ? xr : 0);
        const int64_t y0 = y[0] + (k == 0 ? yr : 0), y1 = y[1] + (k == 1 ? yr : 0);
        part[k] = max64(max64(2 * x0, 2 * x1), max64(W + y0, W + y1));
      }
      const int k = part[1] < part[0] || (part[1] == part[0] && cnt[1] < cnt[0]) ? 1 : 0;
      seeds[2].g[r] = k;
      x[k] += xr;
      y[k] += yr;
      ++cnt[k];
    }
    if (cnt[0] == 0 || cnt[1] == 0) seeds[2].g[order[n - 1]] ^= 1;  // keep both groups non-empty
  }
  const int64_t max_steps = 64 * (int64_t)n + 1024;
  int best_i = -1;
  int64_t best = INT64_MAX, best_ph = INT64_MAX;
  for (int i = 0; i < 3; ++i) {
    sums_of(seeds[i], cost, n);
    descend(seeds[i], cost, n, D, S, V, max_steps);
    const int64_t t = period2(seeds[i].dA, seeds[i].sA, seeds[i].vA, D, S, V);
    const int64_t ph = phase_max(seeds[i].dA, seeds[i].vA, D, V);
    if (better(t, ph, best, best_ph)) {
      best = t;
      best_ph = ph;
      best_i = i;
    }
  }
  const std::vector<int32_t>& g = seeds[best_i].g;
  const int32_t flip = g[0];  // T(A) = T(B): name the group of request 0 A
  for (int32_t r = 0; r < n; ++r) group[r] = g[r] ^ flip;
  if (period_ns) *period_ns = (best + 1) / 2;
  return VC_OK;
}
