// planner.cpp -- owner placement: whole matrices to owner ranks, host only.
//
// DMuon technical summary (gist.science 2606.27153), §2.3 "compute-aware load
// balancing": each 2-D matrix is updated by exactly one owner rank; the
// assignment minimises the predicted makespan (the largest per-owner cost),
// exactly where the search is small and by a greedy heuristic otherwise.  The
// greedy used here is longest-processing-time first (LPT); the exact search is
// a depth-first branch and bound seeded with the LPT answer.
//
// Both are deterministic functions of (cost, world): every rank computes the
// same placement locally, so placement needs no communication.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

#include "muon_ns.h"

namespace muon {

muon_status fail(muon_status s, const char* fmt, ...);

namespace {

// Matrices in order of decreasing cost; equal costs keep input order.
std::vector<int> by_cost(const double* cost, int count) {
  std::vector<int> ord(count);
  std::iota(ord.begin(), ord.end(), 0);
  std::stable_sort(ord.begin(), ord.end(), [&](int x, int y) { return cost[x] > cost[y]; });
  return ord;
}

// Greedy LPT: each matrix, heaviest first, goes to the least-loaded owner
// (lowest rank among equal loads).
double lpt(const double* cost, int count, int world, const std::vector<int>& ord, int32_t* owner,
           std::vector<double>& load) {
  load.assign(world, 0.0);
  for (int i : ord) {
    int r = 0;
    for (int q = 1; q < world; ++q)
      if (load[q] < load[r]) r = q;
    owner[i] = r;
    load[r] += cost[i];
  }
  return *std::max_element(load.begin(), load.end());
}

struct Search {
  const double* cost;
  const std::vector<int>* ord;
  int count, world;
  std::vector<double> load;
  std::vector<int32_t> cur;
  std::vector<int32_t> best;
  double best_span;
  double bound;  // no assignment can beat this: max(max cost, total / world)
  long long nodes, budget;
  bool done;

  void dfs(int t, double span) {
    if (done) return;
    if (++nodes > budget) {
      done = true;
      return;
    }
    if (t == count) {
      if (span < best_span) {
        best_span = span;
        best = cur;
        if (best_span <= bound) done = true;
      }
      return;
    }
    const int i = (*ord)[t];
    for (int r = 0; r < world; ++r) {
      // owners with equal load are interchangeable: try only the first of them
      bool seen = false;
      for (int q = 0; q < r && !seen; ++q) seen = load[q] == load[r];
      if (seen) continue;
      const double nl = load[r] + cost[i];
      const double ns = std::max(span, nl);
      if (ns >= best_span) continue;  // cannot improve on the best found
      load[r] = nl;
      cur[i] = r;
      dfs(t + 1, ns);
      load[r] -= cost[i];
      if (done) return;
    }
  }
};

}  // namespace
}  // namespace muon

using namespace muon;

extern "C" {

muon_status muon_partition(const double* cost, int count, int world, int exact_limit, int32_t* owner,
                           double* load_out) {
  if (count < 0) return fail(MUON_ERR_ARG, "count=%d < 0", count);
  if (world < 1) return fail(MUON_ERR_ARG, "world=%d < 1", world);
  if (count > 0 && (!cost || !owner)) return fail(MUON_ERR_ARG, "cost and owner must not be NULL");
  if (exact_limit < 0 || exact_limit > MUON_PARTITION_EXACT_MAX)
    return fail(MUON_ERR_ARG, "exact_limit=%d out of [0, %d]", exact_limit, MUON_PARTITION_EXACT_MAX);
  for (int i = 0; i < count; ++i)
    if (!(std::isfinite(cost[i]) && cost[i] >= 0.0))
      return fail(MUON_ERR_ARG, "cost[%d] must be finite and non-negative", i);
  std::vector<double> load;
  const std::vector<int> ord = by_cost(cost, count);
  double span = lpt(cost, count, world, ord, owner, load);
  if (count > 0 && count <= exact_limit && world > 1) {
    Search s;
    s.cost = cost;
    s.ord = &ord;
    s.count = count;
    s.world = world;
    s.load.assign(world, 0.0);
    s.cur.assign(count, 0);
    s.best.assign(owner, owner + count);
    s.best_span = span;
    const double total = std::accumulate(cost, cost + count, 0.0);
    s.bound = std::max(cost[ord[0]], total / world);
    s.nodes = 0;
    s.budget = MUON_PARTITION_NODE_BUDGET;
    s.done = span <= s.bound;
    s.dfs(0, 0.0);
    if (s.best_span < span) {
      std::copy(s.best.begin(), s.best.end(), owner);
      load.assign(world, 0.0);
      for (int i = 0; i < count; ++i) load[owner[i]] += cost[i];
    }
  }
  if (load_out)
    for (int r = 0; r < world; ++r) load_out[r] = r < static_cast<int>(load.size()) ? load[r] : 0.0;
  return MUON_OK;
}

}  // extern "C"
