"""Balance scheduler of the ByteScale research digest (section 3.4, Figure 4),
written out as plain Python loops over integers.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Shares no code with
the library's C++ implementation.

The section states the steps but not Algorithm 2's text; the reading taken
here (and in the library) is:
  1. order the micro-batches by cost, heaviest first (ties: lower index first);
  2. cut that order into B consecutive buckets of about equal total cost: the
     item at sorted position p goes to bucket min(B-1, floor(B * P_p / total)),
     P_p being the cost of the items before it (all in bucket 0 if total = 0);
  3. DP-Balance: all workers draw from the front of that order, i.e. from the
     first non-empty bucket, so they work on one length level at a time.  In
     each pass every worker whose load trails the slowest worker's load by
     more than delta takes the next micro-batch (in worker order); when no
     worker trails by more than delta, every worker takes one;
     PP-Balance: with one bucket per pipeline, pipeline p takes bucket p, so
     pipelines of heavier micro-batches get fewer of them and the bucket
     totals (about equal) are their loads.
Costs are the per-micro-batch useful FLOPs (section 2), exact integers.
"""
from __future__ import annotations

DP, PP = 0, 1


def buckets_of(costs, num_buckets: int):
    """Steps 1-2: (sorted order, bucket of each item by item index)."""
    m = len(costs)
    order = sorted(range(m), key=lambda i: (-int(costs[i]), i))
    total = sum(int(c) for c in costs)
    bucket = [0] * m
    before = 0
    for i in order:
        b = 0 if total == 0 else min(num_buckets - 1, (num_buckets * before) // total)
        bucket[i] = b
        before += int(costs[i])
    return order, bucket


def schedule(costs, workers: int, num_buckets: int, delta: int, mode: int = DP):
    """Returns (worker of each item, load of each worker, bucket of each item)."""
    m = len(costs)
    if mode == PP:
        num_buckets = workers
    order, bucket = buckets_of(costs, num_buckets)
    worker_of = [-1] * m
    load = [0] * workers
    if mode == PP:
        for i in range(m):
            worker_of[i] = bucket[i]
            load[bucket[i]] += int(costs[i])
        return worker_of, load, bucket
    pos = 0
    while pos < m:
        slowest = max(load)
        trailing = [w for w in range(workers) if load[w] + delta < slowest]
        if not trailing:
            trailing = list(range(workers))
        for w in trailing:
            if pos == m:
                break
            i = order[pos]
            pos += 1
            worker_of[i] = w
            load[w] += int(costs[i])
    return worker_of, load, bucket
