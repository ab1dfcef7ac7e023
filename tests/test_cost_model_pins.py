"""Pins of the cost-model oracle (``oracle/cost_model.py``) to what the pages
and the mathematics fix, independent of the oracle's own formulas:

- the worked cases printed in the ByteScale research digest, section 3.2
  (``tests/golden/ring_model_worked_cases.json``): 255 x 1.5 + 0.35 ~ 383 ms,
  39 x 2.8 ~ 109 ms, both within 6% of the measured 405 / 110 ms, and the
  static ring hiding its transfers only from about 1.1M tokens;
- closed forms the section derives: a sequence filling the ring gives
  t_c = t_blk; a pack of equal-length sequences gives t_c = t_blk s / S_max;
- the two readings of Eq. 3 stated in section 3.3 (r = 0 gives D ~ s/C,
  r = 1 gives D ~ 2s/(lC)) and a brute-force minimisation over r;
- least squares: exact recovery of noiseless polynomials and the normal
  equations on noisy data.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import cost_model as cm

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "ring_model_worked_cases.json")))


def test_static_ring_worked_case():
    g = GOLD["static_ring"]
    assert g["context_tokens"] // g["ranks"] == g["tokens_per_rank"] == GOLD["capacity_tokens"]
    t = cm.ring_attention_time(g["ranks"], g["t_c_ms"], g["t_x_ms"])
    assert t == pytest.approx(255 * 1.5 + 0.35, abs=1e-9)
    assert round(t) == g["model_ms_printed"]
    assert abs(t - g["measured_ms"]) / g["measured_ms"] <= GOLD["model_vs_measured_within"]


def test_hdp_ring_worked_case():
    g = GOLD["hdp_ring"]
    assert g["sequence_tokens"] // g["ranks"] == g["tokens_per_rank"] == GOLD["capacity_tokens"]
    t_c = cm.ring_step_compute([g["sequence_tokens"]], g["ranks"], GOLD["capacity_tokens"], g["t_blk_ms"])
    assert t_c == pytest.approx(g["t_blk_ms"], rel=1e-15)  # one sequence fills the ring
    t = cm.ring_attention_time(g["ranks"], t_c, g["t_x_ms"])
    assert t == pytest.approx(39 * 2.8, rel=1e-12)
    assert round(t) == g["model_ms_printed"]
    assert abs(t - g["measured_ms"]) / g["measured_ms"] <= GOLD["model_vs_measured_within"]


def test_p2p_share_worked_case():
    g = GOLD["p2p_share"]
    assert round(g["attention_ms"] / (g["attention_ms"] + g["mlp_ms"]), 3) == g["share_printed"]


def test_equal_length_pack_closed_form_and_hide_threshold():
    C, N = GOLD["capacity_tokens"], 256
    s_max = N * C
    t_blk, t_x = 2.8, 1.5
    for s in (1024, 8192, 65536, 262144, 1048576, 2097152):
        k = s_max // s
        t_c = cm.ring_step_compute([s] * k, N, C, t_blk)
        assert t_c == pytest.approx(t_blk * s / s_max, rel=1e-13)
    # shortest hidden length: the first s whose pack computes at least t_x per step
    s_star = math.ceil(t_x / t_blk * s_max)
    g = GOLD["static_ring_hide"]
    assert abs(s_star - g["shortest_hidden_printed_tokens"]) / g["shortest_hidden_printed_tokens"] < 0.05
    # the model agrees on packs of equal lengths that divide S_max: 1M-token
    # sequences (2 per pack) leave the ring waiting, 2M (1 per pack) hide
    assert cm.ring_step_compute([1 << 20] * 2, N, C, t_blk) < t_x
    assert cm.ring_step_compute([1 << 21], N, C, t_blk) >= t_x
    assert (1 << 20) < s_star <= (1 << 21)


def test_ring_time_special_cases():
    assert cm.ring_attention_time(1, 0.7, 5.0) == 0.7      # one rank: no transfer
    assert cm.ring_attention_time(4, 2.0, 1.0) == 8.0      # compute-bound: N t_c
    assert cm.ring_attention_time(4, 1.0, 2.0) == 7.0      # transfer-bound
    # t_c is additive over sequences and quadratic in each
    a = cm.ring_step_compute([100], 4, 1000, 1.0)
    b = cm.ring_step_compute([200], 4, 1000, 1.0)
    assert b == pytest.approx(4 * a, rel=1e-15)
    assert cm.ring_step_compute([100, 200], 4, 1000, 1.0) == pytest.approx(a + b, rel=1e-15)


def _model(**kw):
    m = dict(alpha1=1e-9, beta1=1e-5, gamma=0.1, alpha2=2.0, beta2=0.0, bw_d2h=1e6, bw_h2d=1e6, layers=8)
    m.update(kw)
    return m


def test_eq3_no_offload_reading():
    """r = 0 gives D = ceil(s / C) when Act is proportional to s (section 3.3)."""
    C = 8192
    for s in (1, 8191, 8192, 8193, 100000, 2097152, 3 * 8192):
        r, d = cm.offload_ranks(_model(bw_d2h=0.0), s, C)
        assert r == 0.0
        assert d == math.ceil(s / C)


def test_eq3_full_offload_reading():
    """r = 1 gives D = ceil(2 s / (l C)) (section 3.3) when the copy hides."""
    C = 8192
    for l in (3, 4, 8, 32):
        for s in (65536, 300000, 2097152):
            r, d = cm.offload_ranks(_model(layers=l, bw_d2h=1e30, bw_h2d=1e30), s, C)
            assert r == 1.0
            assert d == math.ceil(2 * s / (l * C))


def test_eq3_matches_brute_force_minimisation():
    rng = np.random.default_rng(3)
    C = 8192
    for _ in range(200):
        l = int(rng.integers(3, 40))
        s = int(rng.integers(1, 4_000_000))
        m = _model(alpha1=float(rng.uniform(1e-10, 1e-8)), beta1=float(rng.uniform(0, 1e-4)),
                   gamma=float(rng.uniform(0, 1.0)), alpha2=float(rng.uniform(0.5, 4.0)),
                   beta2=float(rng.uniform(0, 1e4)), bw_d2h=float(rng.uniform(0, 5e5)),
                   bw_h2d=float(rng.uniform(0, 5e5)), layers=l)
        r, d = cm.offload_ranks(m, s, C)
        act = lambda x: m["alpha2"] * x + m["beta2"]
        t = m["alpha1"] * s * s + m["beta1"] * s + m["gamma"]
        r_lo = min(1.0, l * act(C) / ((l - 2) * act(s)))
        r_hide = t * min(m["bw_d2h"], m["bw_h2d"]) / act(s)
        best = math.ceil(act(s) / act(C) - 1e-12)  # r = 0 is always allowed
        # the admissible set is [r_lo, min(1, r_hide)]: a grid plus both ends
        cands = list(np.linspace(r_lo, 1.0, 257)) + [min(1.0, r_hide)]
        for rr in cands:
            if r_lo <= rr <= r_hide:
                best = min(best, math.ceil((2 * act(s) + (1 - rr) * (l - 2) * act(s)) / (l * act(C)) - 1e-12))
        assert d == best, (s, l, r, d, best)
        assert 0.0 <= r <= 1.0


@pytest.mark.parametrize("degree", [1, 2])
def test_fit_recovers_noiseless_polynomials(degree):
    rng = np.random.default_rng(degree)
    x = np.array([2048, 4096, 8192, 16384, 32768, 65536, 131072], dtype=np.float64)
    true = [0.05, 3e-6, 4e-11][: degree + 1]
    y = sum(c * x**k for k, c in enumerate(true))
    coef = cm.fit_cost_model(x, y, degree)
    for k in range(degree + 1):
        assert coef[k] == pytest.approx(true[k], rel=1e-7, abs=1e-12)
    perm = rng.permutation(len(x))
    assert np.allclose(cm.fit_cost_model(x[perm], y[perm], degree), coef, rtol=1e-9, atol=0)


def test_fit_satisfies_normal_equations():
    rng = np.random.default_rng(7)
    x = rng.uniform(1, 100, 50)
    y = 0.3 * x**2 - 2 * x + 5 + rng.normal(0, 1, 50)
    coef = cm.fit_cost_model(x, y, 2)
    v = np.vander(x, 3, increasing=True)
    resid = y - v @ coef
    assert np.max(np.abs(v.T @ resid)) <= 1e-8 * np.max(np.abs(v.T @ y))


def test_weighted_fit_recovers_and_satisfies_weighted_normal_equations():
    x = np.array([2048, 4096, 8192, 16384, 32768, 65536, 131072], dtype=np.float64)
    y = 4e-9 * x**2 + 2e-5 * x + 0.05
    w = 1.0 / y**2
    coef = cm.fit_cost_model(x, y, 2, w)
    assert np.allclose(coef, [0.05, 2e-5, 4e-9], rtol=1e-7, atol=0)
    rng = np.random.default_rng(9)
    yn = y * (1 + rng.normal(0, 0.05, x.size))
    coef = cm.fit_cost_model(x, yn, 2, w)
    v = np.vander(x, 3, increasing=True)
    g = v.T @ (w * (yn - v @ coef))
    assert np.all(np.abs(g) <= 1e-8 * (v.T @ (w * np.abs(yn))))
    # a zero weight removes a point: same fit as without it
    w2 = w.copy()
    w2[3] = 0.0
    keep = np.arange(x.size) != 3
    assert np.allclose(cm.fit_cost_model(x, yn, 2, w2), cm.fit_cost_model(x[keep], yn[keep], 2, w[keep]),
                       rtol=1e-9, atol=0)
