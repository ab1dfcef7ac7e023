"""Parity of the library's balance scheduler (host C++ in libhdpattn.so,
through the C ABI) with the oracle: bit-exact placements, loads and buckets
on seeded inputs, including the shard FLOPs of the named workloads' plans
(computed by the oracle).  No GPU is needed."""
import numpy as np
import pytest

import oracle
import packed_varlen_attention_aware_gb300 as pkg
from oracle import balance as bal
from packed_varlen_attention_aware_gb300 import workloads as wl


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from packed_varlen_attention_aware_gb300 import build

    build.build()


def _compare(costs, R, B, delta, mode):
    w, load, b = pkg.hdp_balance_schedule(costs, R, B, delta, mode)
    w_ref, load_ref, b_ref = bal.schedule([int(c) for c in costs], R, B, delta, mode)
    assert w.tolist() == w_ref
    assert load.tolist() == load_ref
    assert b.tolist() == b_ref


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("mode", [pkg.HDP_BALANCE_DP, pkg.HDP_BALANCE_PP])
def test_random(seed, mode):
    rng = np.random.default_rng(100 + seed)
    m = int(rng.integers(0, 600))
    scale = int(rng.choice([10, 10**6, 10**15]))
    costs = rng.integers(0, scale, m, dtype=np.int64)
    if seed % 3 == 0 and m:
        costs[: m // 2] = costs[0]  # many ties
    R, B = int(rng.integers(1, 70)), int(rng.integers(1, 20))
    delta = int(rng.integers(0, scale))
    _compare(costs, R, B, delta, mode)


@pytest.mark.parametrize("name", ["mb32k", "mix1m", "seq2m"])
def test_named_workload_shards(name):
    w = wl.workload(name)
    ref = oracle.plan(np.array(w.lengths, dtype=np.int32), w.capacity)
    costs = oracle.flops_per_shard(ref, w.d, w.hq)
    for R in (1, 4, 16, 64):
        for delta in (0, int(np.max(costs)) // 8):
            _compare(costs, R, 4, delta, pkg.HDP_BALANCE_DP)
        _compare(costs, R, 4, 0, pkg.HDP_BALANCE_PP)


def test_argument_errors():
    E = pkg.HdpError
    with pytest.raises(E):
        pkg.hdp_balance_schedule([1, -1], 2, 1, 0)
    with pytest.raises(E):
        pkg.hdp_balance_schedule([1], 0, 1, 0)
    with pytest.raises(E):
        pkg.hdp_balance_schedule([1], 1, 0, 0)
    with pytest.raises(E):
        pkg.hdp_balance_schedule([1], 1, 1, -1)
    with pytest.raises(E):
        pkg.hdp_balance_schedule([2**62, 2**62], 1, 1, 0)  # total overflows int64
    w, load, b = pkg.hdp_balance_schedule([], 3, 2, 0)
    assert w.size == 0 and load.tolist() == [0, 0, 0]
