"""Pins for the oracle's fp32 fixed-point decision arithmetic (CPU only).

The recipe (E = Cody-Waite + degree-7 Taylor exp, L = exponent + atanh-series
log, Q = floor(2^40 E(s - m))) is checked against the exact functions within
the error bound of the method, and against closed forms.
"""
import math

import numpy as np
import pytest

import oracle


def ulp32(x: float) -> float:
    return float(np.spacing(np.float32(abs(x))))


def test_exp_recipe_within_2ulp_of_exact():
    xs = np.concatenate([np.linspace(-32.0, 0.0, 200_001, dtype=np.float32),
                         -np.geomspace(1e-8, 32.0, 20_001).astype(np.float32)])
    worst = 0.0
    for x in xs[::7]:
        e = oracle.exp_recipe(float(x))
        ref = math.exp(float(x))
        err = abs(e - ref) / ulp32(ref)
        worst = max(worst, err)
    assert worst <= 2.0, worst


def test_exp_recipe_special_values():
    assert oracle.exp_recipe(0.0) == 1.0
    assert oracle.exp_recipe(-33.0) == 0.0
    assert abs(oracle.exp_recipe(-math.log(2.0)) - 0.5) <= ulp32(0.5)


def test_qmass_closed_forms():
    # the row maximum carries exactly 2^40
    for m in [0.0, 3.5, -7.25, 1e4]:
        assert oracle.qmass(m, m) == 2 ** 40
    # exp(-ln 2) = 1/2  ->  2^39 within one fp32 ulp of the scaled value
    s = float(np.float32(-math.log(2.0)))
    assert abs(oracle.qmass(s, 0.0) - 2 ** 39) <= 2 ** 39 * 2 ** -23
    # below 2^-40 the mass is zero
    assert oracle.qmass(-28.0, 0.0) == 0
    # monotone in s
    prev = 0
    for s in np.linspace(-27.0, 0.0, 5001, dtype=np.float32):
        q = oracle.qmass(float(s), 0.0)
        assert q >= prev
        prev = q


def test_ell_recipe_matches_log():
    assert oracle.ell(2 ** 40) == 0.0
    rng = np.random.default_rng(7)
    Qs = [2 ** 40, 2 ** 41, 3 * 2 ** 40, 2 ** 57 - 1] + [int(x) for x in rng.integers(2 ** 40, 2 ** 57, 5000)]
    for Q in Qs:
        got = oracle.ell(Q)
        ref = math.log(Q) - 40 * math.log(2.0)
        # fp32 conversion of Q (2^-24 rel) + a few ulp of the result
        assert abs(got - ref) <= 2 ** -23 + 4 * ulp32(ref), (Q, got, ref)
        assert got >= 0.0


def test_row_stats_against_exact_softmax():
    rng = np.random.default_rng(11)
    z = (rng.standard_normal((6, 3000)) * 4).astype(np.float32)
    z[2, 17] = z[2, 5] = z[2].max() + 1.0  # a tie for the argmax -> lowest id
    T = np.array([1.0, 0.7, 1.0, 0.0, -1.0, 2.0], np.float32)
    m, Q, am, bad = oracle.row_stats(z, T)
    assert not bad.any()
    for i in range(6):
        it = np.float32(1.0) / T[i] if T[i] > 0 else np.float32(1.0)
        s = (z[i] * it).astype(np.float32)
        assert m[i] == s.max()
        assert am[i] == int(np.flatnonzero(s == s.max())[0])
        exact = sum(math.floor(math.exp(float(v) - float(m[i])) * 2 ** 40) for v in s)
        assert abs(int(Q[i]) - exact) <= 1e-6 * exact + len(s)
    assert am[2] == 5


def test_row_stats_flags_nonfinite():
    z = np.zeros((3, 10), np.float32)
    z[1, 3] = np.nan
    z[2, 9] = np.inf
    _, _, _, bad = oracle.row_stats(z, 1.0)
    assert list(bad) == [0, 1, 1]
