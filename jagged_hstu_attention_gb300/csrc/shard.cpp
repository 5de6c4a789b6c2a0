// Host-only partitioning of a jagged batch over data-parallel ranks.
//
// Every (sequence, head) unit of the attention op is independent in both the
// forward and the backward pass, and dq/dk/dv are per token, so a batch can
// be split by whole sequences with no exchange between ranks. The split is
// the greedy longest-processing-time rule (Graham, "Bounds on multiprocessing
// timing anomalies", 1969): sequences in descending cost each go to the rank
// whose load is smallest so far. Its makespan is at most (4/3 - 1/(3W)) times
// the optimum for W ranks.

#include <algorithm>
#include <numeric>
#include <queue>
#include <vector>

#include "hstu_attn.h"

namespace {

struct RankLoad {
  int64_t load;
  int32_t rank;
};

// Orders the priority queue so that top() is the least-loaded rank, the
// lower rank first among equal loads.
struct HeavierFirst {
  bool operator()(const RankLoad& a, const RankLoad& b) const {
    return a.load != b.load ? a.load > b.load : a.rank > b.rank;
  }
};

}  // namespace

extern "C" HSTU_API hstu_status_t hstu_attn_shard_sequences(const int64_t* cost, int32_t batch,
                                                            int32_t world, int32_t* owner,
                                                            int64_t* rank_load) {
  if (batch < 0 || world < 1 || (batch > 0 && (cost == nullptr || owner == nullptr)))
    return HSTU_ERR_INVALID_ARG;
  int64_t total = 0;
  for (int32_t i = 0; i < batch; ++i) {
    if (cost[i] < 0 || __builtin_add_overflow(total, cost[i], &total)) return HSTU_ERR_INVALID_ARG;
  }
  try {
    std::vector<int32_t> order(static_cast<size_t>(batch));
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(),
                     [cost](int32_t a, int32_t b) { return cost[a] > cost[b]; });
    std::priority_queue<RankLoad, std::vector<RankLoad>, HeavierFirst> ranks;
    for (int32_t r = 0; r < world; ++r) ranks.push({0, r});
    std::vector<int64_t> load(static_cast<size_t>(world), 0);
    for (int32_t i : order) {
      RankLoad r = ranks.top();
      ranks.pop();
      owner[i] = r.rank;
      r.load += cost[i];  // no overflow: every partial sum is at most total
      load[r.rank] = r.load;
      ranks.push(r);
    }
    if (rank_load != nullptr) std::copy(load.begin(), load.end(), rank_load);
  } catch (...) {  // allocation failure; no exception crosses the C ABI
    return HSTU_ERR_INVALID_ARG;
  }
  return HSTU_OK;
}
