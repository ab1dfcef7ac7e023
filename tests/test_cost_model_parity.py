"""Parity of the library's cost-model calls (host arithmetic in libhdpattn.so,
reached through the C ABI) with the exact-rational oracle, on seeded random
inputs and on the edge cases each call documents.  No GPU is needed: these
entry points touch no device.
"""
import math

import numpy as np
import pytest

import packed_varlen_attention_aware_gb300 as pkg
from oracle import cost_model as cm


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from packed_varlen_attention_aware_gb300 import build

    build.build()


def test_ring_step_compute_matches_oracle():
    rng = np.random.default_rng(0)
    for _ in range(300):
        N = int(rng.integers(1, 512))
        C = int(rng.choice([1024, 4096, 8192, 32768]))
        n = int(rng.integers(1, 64))
        lengths = rng.integers(1, max(2, N * C // n), n)
        lengths = lengths[: max(1, np.searchsorted(np.cumsum(lengths), N * C, side="right"))]
        if lengths.sum() > N * C:
            lengths = np.array([N * C])
        t_blk = float(rng.uniform(0.01, 10))
        got = pkg.hdp_ring_step_compute(lengths, N, C, t_blk)
        assert got == pytest.approx(cm.ring_step_compute(lengths, N, C, t_blk), rel=1e-15, abs=0)


def test_ring_attention_time_matches_oracle():
    rng = np.random.default_rng(1)
    for _ in range(300):
        N = int(rng.integers(1, 100000))
        t_c, t_x = (float(v) for v in rng.uniform(0, 5, 2))
        assert pkg.hdp_ring_attention_time(N, t_c, t_x) == pytest.approx(cm.ring_attention_time(N, t_c, t_x),
                                                                          rel=1e-15, abs=0)


def _rand_model(rng):
    return dict(alpha1=float(rng.uniform(1e-10, 1e-8)), beta1=float(rng.uniform(0, 1e-4)),
                gamma=float(rng.uniform(0, 1.0)), alpha2=float(rng.uniform(0.5, 4.0)),
                beta2=float(rng.uniform(0, 1e4)), bw_d2h=float(rng.uniform(0, 5e5)),
                bw_h2d=float(rng.uniform(0, 5e5)), layers=int(rng.integers(3, 64)))


def test_offload_ranks_matches_oracle():
    rng = np.random.default_rng(2)
    for _ in range(2000):
        m = _rand_model(rng)
        s = int(rng.integers(1, 8_000_000))
        C = int(rng.choice([2048, 8192, 65536]))
        r, d = pkg.hdp_offload_ranks(m, s, C)
        r_ref, d_ref = cm.offload_ranks(m, s, C)
        assert d == d_ref, (m, s, C)
        assert r == pytest.approx(r_ref, rel=1e-12, abs=1e-15)


def test_offload_ranks_exact_multiples_not_pushed_up():
    # Act(s) = 0.1 s (0.1 is not a binary fraction): r = 0 must give exactly s / C
    m = dict(alpha1=0.0, beta1=0.0, gamma=0.0, alpha2=0.1, beta2=0.0, bw_d2h=0.0, bw_h2d=0.0, layers=7)
    for k in range(1, 300):
        r, d = pkg.hdp_offload_ranks(m, k * 8192, 8192)
        assert (r, d) == (0.0, k)


@pytest.mark.parametrize("degree", [1, 2])
def test_fit_matches_oracle(degree):
    rng = np.random.default_rng(10 + degree)
    for _ in range(50):
        n = int(rng.integers(degree + 1, 40))
        x = rng.uniform(256, 2_097_152, n)
        coef_true = [rng.uniform(0, 1), rng.uniform(0, 1e-4), rng.uniform(0, 1e-9)][: degree + 1]
        y = sum(c * x**k for k, c in enumerate(coef_true)) * (1 + rng.normal(0, 0.01, n))
        w = None if _ % 2 else rng.uniform(0, 2, n) / np.maximum(y, 1e-30) ** 2
        got = pkg.hdp_fit_cost_model(x, y, degree, w)
        ref = cm.fit_cost_model(x, y, degree, w)
        # compare the fitted curves over the sampled range (coefficients of an
        # ill-conditioned basis can differ more than the curves do)
        xs = np.linspace(x.min(), x.max(), 64)
        fg = sum(c * xs**k for k, c in enumerate(got))
        fr = sum(c * xs**k for k, c in enumerate(ref))
        assert np.max(np.abs(fg - fr)) <= 1e-9 * np.max(np.abs(fr))


def test_argument_errors():
    E = pkg.HdpError
    with pytest.raises(E):
        pkg.hdp_ring_step_compute([0], 1, 8, 1.0)          # length < 1
    with pytest.raises(E):
        pkg.hdp_ring_step_compute([9], 1, 8, 1.0)          # pack larger than the ring
    with pytest.raises(E):
        pkg.hdp_ring_step_compute([4], 0, 8, 1.0)
    with pytest.raises(E):
        pkg.hdp_ring_attention_time(0, 1.0, 1.0)
    with pytest.raises(E):
        pkg.hdp_ring_attention_time(2, -1.0, 1.0)
    m = dict(alpha1=0.0, beta1=0.0, gamma=0.0, alpha2=1.0, beta2=0.0, bw_d2h=1.0, bw_h2d=1.0, layers=2)
    with pytest.raises(E):
        pkg.hdp_offload_ranks(m, 100, 10)                  # layers < 3
    m["layers"] = 4
    m["alpha2"] = 0.0
    with pytest.raises(E):
        pkg.hdp_offload_ranks(m, 100, 10)                  # Act(C) = 0
    with pytest.raises(E):
        pkg.hdp_fit_cost_model([1.0, 1.0, 1.0], [1.0, 2.0, 3.0], 2)   # one distinct x
    with pytest.raises(E):
        pkg.hdp_fit_cost_model([1.0, 2.0], [1.0, 2.0], 2)             # n <= degree
    with pytest.raises(E):
        pkg.hdp_fit_cost_model([1.0, 2.0, math.nan], [1.0, 2.0, 3.0], 1)
    with pytest.raises(E):
        pkg.hdp_fit_cost_model([1.0, 2.0, 3.0], [1.0, 2.0, 3.0], 1, w=[1.0, -1.0, 1.0])
    with pytest.raises(E):
        pkg.hdp_fit_cost_model([1.0, 2.0, 3.0], [1.0, 2.0, 3.0], 1, w=[1.0, 0.0, 0.0])  # one weighted x
