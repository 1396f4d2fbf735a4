// AssignGrid: placement of replay units on a grid of replay rounds x replay lanes.
//
// AugTree paper, Sec. 3.4 ("Replay units and grid assignment", Eq. 6): every replay
// unit k (one complete response path, work estimate w_k) is placed on one cell
// (round tau_k, lane j_k) of a b x s grid; a lane runs its rounds one after another,
// and the placement minimises the replay critical path, the largest lane total
// max_j sum_{k: j_k = j} w_k.  The pages solve it exactly by a bounded subset dynamic
// program when the unit count U is at most a small cap U_max, and by largest-first
// greedy balancing otherwise.  Each cell holds at most one unit, so a lane takes at
// most b units.
//
// Host-only code: no device memory, no CUDA calls.
#include <algorithm>
#include <cstdint>
#include <limits>
#include <new>
#include <numeric>
#include <vector>

#include "augtree.h"

namespace {

constexpr int kMaxExactUnits = 16;  // 3^16 / 2 subset steps per lane level at most
constexpr int64_t kInf = std::numeric_limits<int64_t>::max();

// Units in largest-first order: weight descending, then index ascending.
std::vector<int> largest_first(const int64_t* w, int n) {
  std::vector<int> order(n);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return w[a] > w[b]; });
  return order;
}

// Rounds within each lane: the lane's units in largest-first order take rounds
// 0, 1, 2, ...
void number_rounds(const int64_t* w, int n, const int32_t* lane, int lanes, int32_t* round) {
  std::vector<int32_t> used(lanes, 0);
  for (int k : largest_first(w, n)) round[k] = used[lane[k]]++;
}

int64_t lane_makespan(const int64_t* w, int n, const int32_t* lane, int lanes) {
  std::vector<int64_t> load(lanes, 0);
  for (int k = 0; k < n; ++k) load[lane[k]] += w[k];
  return n ? *std::max_element(load.begin(), load.end()) : 0;
}

// Largest-first greedy: each unit, in largest-first order, goes to the lane with the
// smallest load among those with a free round, ties to the lowest lane index.
void assign_lpt(const int64_t* w, int n, int rounds, int lanes, int32_t* lane) {
  std::vector<int64_t> load(lanes, 0);
  std::vector<int32_t> used(lanes, 0);
  for (int k : largest_first(w, n)) {
    int best = -1;
    for (int j = 0; j < lanes; ++j)
      if (used[j] < rounds && (best < 0 || load[j] < load[best])) best = j;
    lane[k] = best;
    load[best] += w[k];
    ++used[best];
  }
}

// Exact subset DP over lanes.  F_j(M) = the smallest largest-lane total with which the
// unit set M fits on j lanes of at most `rounds` units each.  Lanes are
// interchangeable, so the lane holding M's lowest unit is taken to be lane j:
//   F_j(M) = min over S with low(M) in S subset of M, |S| <= rounds of
//            max(W(S), F_{j-1}(M \ S)),      F_j(empty) = 0, F_0(M != empty) = inf.
// Lane indices come out in the order the recursion peels the sets off.
void assign_exact(const int64_t* w, int n, int rounds, int lanes, int32_t* lane) {
  const int L = std::min(lanes, n);
  const uint32_t full = (n == 32) ? 0xFFFFFFFFu : ((1u << n) - 1u);
  const size_t M = (size_t)full + 1;
  std::vector<int64_t> W(M, 0);
  std::vector<uint8_t> pc(M, 0);
  for (uint32_t m = 1; m <= full; ++m) {
    const int low = __builtin_ctz(m);
    W[m] = W[m & (m - 1)] + w[low];
    pc[m] = (uint8_t)(pc[m & (m - 1)] + 1);
  }
  std::vector<int64_t> prev(M, kInf), cur(M, kInf);
  prev[0] = 0;
  std::vector<std::vector<uint32_t>> choice(L + 1, std::vector<uint32_t>(M, 0));
  for (int j = 1; j <= L; ++j) {
    cur[0] = 0;
    for (uint32_t m = 1; m <= full; ++m) {
      const uint32_t low = m & (~m + 1u);
      const uint32_t rest = m ^ low;
      int64_t best = kInf;
      uint32_t arg = 0;
      uint32_t sub = rest;
      while (true) {
        const uint32_t S = sub | low;
        if (pc[S] <= rounds) {
          const int64_t other = prev[m ^ S];
          if (other != kInf) {
            const int64_t v = std::max(W[S], other);
            if (v < best) {
              best = v;
              arg = S;
            }
          }
        }
        if (sub == 0) break;
        sub = (sub - 1) & rest;
      }
      cur[m] = best;
      choice[j][m] = arg;
    }
    std::swap(prev, cur);
  }
  uint32_t m = full;
  for (int j = L, l = 0; j >= 1 && m; --j, ++l) {
    const uint32_t S = choice[j][m];
    for (int k = 0; k < n; ++k)
      if (S & (1u << k)) lane[k] = l;
    m ^= S;
  }
}

}  // namespace

extern "C" augtree_status augtree_assign_grid(const int64_t* w, int32_t n_units, int32_t rounds, int32_t lanes,
                                              int32_t u_max, int32_t* round_out, int32_t* lane_out,
                                              int64_t* makespan_out, int32_t* exact_out) {
  if (n_units < 0 || rounds < 1 || lanes < 1 || u_max < 0 || u_max > kMaxExactUnits || !makespan_out)
    return AUGTREE_ERR_INVALID_ARG;
  if (n_units > 0 && (!w || !round_out || !lane_out)) return AUGTREE_ERR_INVALID_ARG;
  if ((int64_t)n_units > (int64_t)rounds * lanes) return AUGTREE_ERR_INVALID_ARG;
  for (int k = 0; k < n_units; ++k)
    if (w[k] < 0) return AUGTREE_ERR_INVALID_ARG;
  const bool exact = n_units <= u_max;
  try {
    if (n_units > 0) {
      if (exact)
        assign_exact(w, n_units, rounds, lanes, lane_out);
      else
        assign_lpt(w, n_units, rounds, lanes, lane_out);
      number_rounds(w, n_units, lane_out, lanes, round_out);
    }
  } catch (const std::bad_alloc&) {
    return AUGTREE_ERR_CAPACITY;
  }
  *makespan_out = lane_makespan(w, n_units, lane_out, lanes);
  if (exact_out) *exact_out = exact ? 1 : 0;
  return AUGTREE_OK;
}
