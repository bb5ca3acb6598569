// Owner assignment of Muon matrices across data-parallel ranks (host only).
//
// DMuon-2, section 3.3 "Load Balancing" and Appendix B "Cost Model and Greedy
// Algorithm for Owner Assignment": every assignment unit u (the Muon
// matrices of one wrapping unit) goes whole to one owner o(u); the objective
// is the NS time of the busiest rank, min max_j sum_{o(u)=j} t_u, subject to
// every rank holding at most (1 + eps) times the average bytes and to the
// units of one layer going to different ranks.  The NS time t_u is measured
// per matrix shape (muon_ns_cost_table), not estimated from element counts.
// The greedy Longest-Processing-Time rule: units sorted by t_u decreasing
// (ties: more elements first, then input order); each unit goes to the rank
// with the smallest accumulated time among the ranks not yet used in its
// layer whose bytes stay under the cap after receiving it; if every such
// rank would exceed the cap, to the one of them with the fewest bytes.  When
// a layer has more units than ranks, every rank is a candidate again.
#include <algorithm>
#include <cmath>
#include <numeric>
#include <vector>

#include "../../include/muon.h"

namespace {

muon_status_t assign(const muon_unit_t* units, int n, int n_ranks, double eps, int32_t* owner) {
  if (n < 0 || n_ranks < 1 || (n > 0 && (!units || !owner)) || !(eps >= 0.0) ||
      !std::isfinite(eps))
    return MUON_ERR_INVALID_ARGUMENT;
  double total_bytes = 0.0;
  for (int i = 0; i < n; ++i) {
    if (!(units[i].cost >= 0.0) || !std::isfinite(units[i].cost) || units[i].bytes < 0 ||
        units[i].elems < 0)
      return MUON_ERR_INVALID_ARGUMENT;
    total_bytes += static_cast<double>(units[i].bytes);
  }
  const double cap = (1.0 + eps) * total_bytes / n_ranks;
  std::vector<int> order(n);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
    if (units[a].cost != units[b].cost) return units[a].cost > units[b].cost;
    if (units[a].elems != units[b].elems) return units[a].elems > units[b].elems;
    return a < b;
  });
  std::vector<double> t(n_ranks, 0.0), by(n_ranks, 0.0);
  // ranks already holding a unit of each layer
  std::vector<std::pair<int32_t, int>> used;   // (layer, rank)
  std::vector<char> in_layer(n_ranks);
  for (int u : order) {
    const muon_unit_t& U = units[u];
    std::fill(in_layer.begin(), in_layer.end(), 0);
    int n_in = 0;
    if (U.layer >= 0)
      for (auto& lr : used)
        if (lr.first == U.layer && !in_layer[lr.second]) {
          in_layer[lr.second] = 1;
          ++n_in;
        }
    const bool spread = n_in < n_ranks;   // some rank is still free in this layer
    int best = -1, fewest = -1;
    for (int r = 0; r < n_ranks; ++r) {
      if (spread && in_layer[r]) continue;
      if (fewest < 0 || by[r] < by[fewest]) fewest = r;
      if (by[r] + static_cast<double>(U.bytes) <= cap && (best < 0 || t[r] < t[best])) best = r;
    }
    const int r = best >= 0 ? best : fewest;
    owner[u] = r;
    t[r] += U.cost;
    by[r] += static_cast<double>(U.bytes);
    if (U.layer >= 0) used.push_back({U.layer, r});
  }
  return MUON_OK;
}

}  // namespace

extern "C" muon_status_t muon_assign_owners(const muon_unit_t* units, int n_units, int n_ranks,
                                            double eps, int32_t* owner_out) {
  try {
    return assign(units, n_units, n_ranks, eps, owner_out);
  } catch (...) {
    return MUON_ERR_OUT_OF_MEMORY;
  }
}
