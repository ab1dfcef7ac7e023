// Balance scheduler of "ByteScale: Communication-Efficient Scaling of LLM
// Training with a 2048K Context Length on 16384 GPUs" (research digest,
// section 3.4 and Figure 4): equal-token micro-batches carry unequal FLOPs,
// so workers run unequal numbers of them.  The section gives the steps
// (heaviest-first equal-FLOP buckets, then work for every worker trailing the
// slowest by more than delta; DP-Balance draws from the first bucket,
// PP-Balance gives each pipeline one bucket) but not Algorithm 2's text; the
// reading implemented is the one stated in include/hdpattn.h.
// Host code, integer arithmetic only: results are exact and deterministic.
#include <algorithm>
#include <cstdint>
#include <new>
#include <vector>

#include "internal.h"

extern "C" hdp_status_t hdp_balance_schedule(const int64_t* costs, int32_t m, int32_t workers, int32_t buckets,
                                             int64_t delta, int32_t mode, int32_t* worker_of_item,
                                             int64_t* worker_load, int32_t* bucket_of_item) {
  if (m < 0 || workers < 1 || buckets < 1 || delta < 0 || (mode != HDP_BALANCE_DP && mode != HDP_BALANCE_PP))
    return hdp::fail(HDP_ERR_INVALID_ARGUMENT,
                     "hdp_balance_schedule: m >= 0, workers >= 1, buckets >= 1, delta >= 0, mode DP or PP");
  if (!worker_load || (m > 0 && (!costs || !worker_of_item)))
    return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_balance_schedule: null pointer");
  int64_t total = 0;
  for (int32_t i = 0; i < m; ++i) {
    if (costs[i] < 0) return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_balance_schedule: negative cost");
    if (costs[i] > INT64_MAX - total)
      return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_balance_schedule: total cost overflows int64");
    total += costs[i];
  }
  const int32_t nb = mode == HDP_BALANCE_PP ? workers : buckets;
  std::vector<int32_t> order;
  try {
    order.resize(static_cast<size_t>(m));
  } catch (const std::bad_alloc&) {
    return hdp::fail(HDP_ERR_OUT_OF_MEMORY, "hdp_balance_schedule: host allocation failed");
  }
  for (int32_t i = 0; i < m; ++i) order[i] = i;
  // 1. heaviest first, ties by index
  std::sort(order.begin(), order.end(), [costs](int32_t a, int32_t b) {
    return costs[a] != costs[b] ? costs[a] > costs[b] : a < b;
  });
  for (int32_t w = 0; w < workers; ++w) worker_load[w] = 0;
  // 2. buckets of about equal cost along that order
  int64_t before = 0;
  for (int32_t p = 0; p < m; ++p) {
    const int32_t i = order[p];
    int32_t b = 0;
    if (total > 0) {
      const __int128 q = static_cast<__int128>(nb) * before / total;
      b = q < nb - 1 ? static_cast<int32_t>(q) : nb - 1;
    }
    if (bucket_of_item) bucket_of_item[i] = b;
    if (mode == HDP_BALANCE_PP) {
      worker_of_item[i] = b;
      worker_load[b] += costs[i];
    }
    before += costs[i];
  }
  if (mode == HDP_BALANCE_PP) return HDP_OK;
  // 3. DP-Balance passes
  int32_t pos = 0;
  while (pos < m) {
    int64_t slowest = worker_load[0];
    for (int32_t w = 1; w < workers; ++w) slowest = std::max(slowest, worker_load[w]);
    bool any = false;
    for (int32_t w = 0; w < workers; ++w) any = any || (worker_load[w] < slowest - delta);
    for (int32_t w = 0; w < workers && pos < m; ++w) {
      // load + delta < slowest, written without overflow
      if (any && !(worker_load[w] < slowest - delta)) continue;
      const int32_t i = order[pos++];
      worker_of_item[i] = w;
      worker_load[w] += costs[i];
    }
  }
  return HDP_OK;
}
