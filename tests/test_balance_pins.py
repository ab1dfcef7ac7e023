"""Pins of the balance-scheduler oracle (``oracle/balance.py``) to what the
pages fix and to hand-worked cases, independent of the oracle's code:

- Figure 4 of the ByteScale research digest (section 3.4): equal-token
  micro-batches of unequal attention time.  Equal counts per rank leave three
  ranks idle; the balance scheduler gives unequal counts and equal time.  The
  figure's workload is reconstructed as one long (cost 5), two medium (3) and
  thirteen short (1) micro-batches on four ranks, which fits its "4 per rank"
  layout and its equal-time result;
- a second case worked by hand with delta > 0 and two buckets;
- special cases: equal costs and an infinite threshold both reduce to
  round-robin over the heaviest-first order; PP-Balance loads are the bucket
  totals, each within one micro-batch of total / B;
- invariants on random inputs (every micro-batch placed once, loads are sums).
"""
import numpy as np
import pytest

from oracle import balance as bal

BIG = 1 << 62


def test_figure4_equal_counts_leave_three_ranks_idle():
    costs = [5, 3, 3] + [1] * 13
    w, load, _ = bal.schedule(costs, 4, 1, BIG)  # never trailing: every pass all ranks take one
    counts = [w.count(r) for r in range(4)]
    assert counts == [4, 4, 4, 4]
    assert load == [8, 6, 6, 4]
    assert sum(1 for x in load if x < max(load)) == 3


def test_figure4_balance_gives_unequal_counts_equal_time():
    costs = [5, 3, 3] + [1] * 13
    w, load, _ = bal.schedule(costs, 4, 1, 0)
    counts = [w.count(r) for r in range(4)]
    # worked by hand: pass 1 gives 5,3,3,1; ranks 1-3 then take short ones
    # while they trail rank 0, until all reach 5; the last four go one each
    assert load == [6, 6, 6, 6]
    assert counts == [2, 4, 4, 6]
    assert max(load) == sum(costs) // 4  # the lower bound total / ranks


def test_hand_worked_delta_and_buckets():
    costs = [7, 4, 4, 3, 2, 2, 1, 1]
    w, load, b = bal.schedule(costs, 3, 2, 1)
    assert b == [0, 0, 0, 1, 1, 1, 1, 1]
    assert w == [0, 1, 2, 1, 2, 0, 1, 2]
    assert load == [9, 8, 7]
    w, load, b = bal.schedule(costs, 2, 0, 0, mode=bal.PP)
    assert w == [0, 0, 0, 1, 1, 1, 1, 1]
    assert load == [15, 9]


def test_order_ties_and_input_order():
    # equal costs: round-robin over index order, counts differ by at most one
    w, load, _ = bal.schedule([6] * 10, 4, 3, 0)
    assert w == [k % 4 for k in range(10)]
    assert load == [18, 18, 12, 12]
    # an infinite threshold is round-robin over the heaviest-first order
    costs = [3, 9, 1, 9, 4]
    w, load, _ = bal.schedule(costs, 2, 1, BIG)
    order = [1, 3, 4, 0, 2]
    assert [w[i] for i in order] == [0, 1, 0, 1, 0]


def test_fewer_items_than_workers_and_zero_costs():
    w, load, _ = bal.schedule([5, 2], 4, 2, 0)
    assert w == [0, 1] and load == [5, 2, 0, 0]
    w, load, b = bal.schedule([0, 0, 0], 2, 3, 0)
    assert b == [0, 0, 0] and load == [0, 0] and w == [0, 1, 0]


@pytest.mark.parametrize("seed", range(5))
def test_invariants_random(seed):
    rng = np.random.default_rng(seed)
    m = int(rng.integers(1, 400))
    costs = [int(c) for c in rng.integers(0, 10**12, m)]
    R, B = int(rng.integers(1, 40)), int(rng.integers(1, 12))
    delta = int(rng.integers(0, 10**11))
    for mode in (bal.DP, bal.PP):
        w, load, b = bal.schedule(costs, R, B, delta, mode)
        nw = R
        assert all(0 <= x < nw for x in w)
        assert [sum(c for c, x in zip(costs, w) if x == r) for r in range(nw)] == load
        assert sum(load) == sum(costs)
        # buckets are contiguous along the heaviest-first order, each within
        # one micro-batch of an equal share
        nb = R if mode == bal.PP else B
        order = sorted(range(m), key=lambda i: (-costs[i], i))
        seq = [b[i] for i in order]
        assert seq == sorted(seq)
        total = sum(costs)
        for k in range(nb - 1):
            tot_k = sum(costs[i] for i in range(m) if b[i] == k)
            if tot_k:
                assert abs(tot_k - total / nb) <= max(costs) + 1
