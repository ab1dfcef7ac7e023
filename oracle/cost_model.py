"""Cost models of the ByteScale research digest, written out in exact rational
arithmetic (Python ``fractions``) so that every quantity is the formula's
value for the given inputs, with no rounding until the final float.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Shares no code with
the library's C++ implementation.

Sources ("ByteScale: Communication-Efficient Scaling of LLM Training with a
2048K Context Length on 16384 GPUs", research digest):
  section 3.2  ring timing model t_c, T_attn and its table of worked cases;
  section 3.3  profiled models T(s), Act(s) and Eq. 3 (offload ratio r and the
               rank count D(s)).
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

# A quotient that lies within this relative distance above an integer counts
# as that integer when Eq. 3 takes its ceiling (the library computes in double
# precision; exact multiples of C must not be pushed up by rounding).
CEIL_REL_TOL = Fraction(1, 10**9)


def _q(x) -> Fraction:
    return Fraction(x)  # exact value of a Python int or float


def ring_step_compute(lengths, num_ranks: int, capacity: int, t_blk: float) -> float:
    """Section 3.2: every sequence s_i of the pack is cut into N slices; a query
    attends only to its own sequence, so one step computes the sum over the
    sequences of (s_i / (N C))^2 full C x C blocks: t_c = t_blk * sum (s_i/(NC))^2."""
    n_c = num_ranks * capacity
    total = sum((Fraction(int(s), n_c) ** 2 for s in lengths), Fraction(0))
    return float(_q(t_blk) * total)


def ring_attention_time(num_ranks: int, t_c: float, t_x: float) -> float:
    """Section 3.2: N - 1 steps that each last max(t_c, t_x), then the last
    compute: T_attn = (N - 1) * max(t_c, t_x) + t_c."""
    tc, tx = _q(t_c), _q(t_x)
    return float((num_ranks - 1) * max(tc, tx) + tc)


def _ceil_tol(x: Fraction) -> int:
    k = math.floor(x)
    if x == k:
        return k
    # within the tolerance above k: counts as k
    if k > 0 and (x - k) <= CEIL_REL_TOL * x:
        return k
    return k + 1


def offload_ranks(model: dict, s: int, capacity: int):
    """Eq. 3 (section 3.3), in the digest's order of the three lines.

    Act(s) = alpha2 s + beta2, T(s) = alpha1 s^2 + beta1 s + gamma.
    Line 3: the admissible ratios are 1 >= r >= min(1, l Act(C) / ((l-2) Act(s))).
    Line 2: the copy must hide behind compute, r <= T(s) min(B_d2h, B_h2d) / Act(s).
    Line 1: D = ceil((2 Act(s) + (1 - r)(l - 2) Act(s)) / (l Act(C))), which does
    not grow with r, so the largest admissible r gives the smallest D; with no
    admissible r the sequence is not offloaded (r = 0).
    Returns (r as float, D as int)."""
    a1, b1, g = _q(model["alpha1"]), _q(model["beta1"]), _q(model["gamma"])
    a2, b2 = _q(model["alpha2"]), _q(model["beta2"])
    bmin = min(_q(model["bw_d2h"]), _q(model["bw_h2d"]))
    l = int(model["layers"])
    act_s = a2 * s + b2
    act_c = a2 * capacity + b2
    t_s = a1 * s * s + b1 * s + g
    r_lo = min(Fraction(1), l * act_c / ((l - 2) * act_s))
    r_hide = t_s * bmin / act_s
    r = min(Fraction(1), r_hide)
    if r < r_lo:
        r = Fraction(0)
    d = _ceil_tol((2 * act_s + (1 - r) * (l - 2) * act_s) / (l * act_c))
    return float(r), int(d)


def fit_cost_model(x, y, degree: int, w=None) -> np.ndarray:
    """Weighted least-squares polynomial through the points (the profiled cost
    models of section 3.3 are fitted this way): minimise sum w_i (y_i - p(x_i))^2;
    coefficients of x^0 .. x^degree.  The solve is numpy's least-squares
    routine on the Vandermonde matrix with rows scaled by sqrt(w_i)."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    w = np.ones_like(x) if w is None else np.asarray(w, dtype=np.float64)
    # change of variable u = x / scale (same minimiser, better conditioned);
    # the coefficient of u^k is the coefficient of x^k times scale^k
    scale = float(np.max(np.abs(x[w > 0])))
    sw = np.sqrt(w)
    v = np.vander(x / scale, degree + 1, increasing=True) * sw[:, None]
    coef_u, *_ = np.linalg.lstsq(v, y * sw, rcond=None)
    return coef_u / scale ** np.arange(degree + 1)
