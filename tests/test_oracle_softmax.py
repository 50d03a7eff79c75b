"""Pins of the row-softmax oracle (oracle/softmax.py) against values fixed by
the mathematics, and planted mistakes each pin set must catch."""

import math
import types

import numpy as np
import pytest

import oracle.softmax as ref

mpmath = pytest.importorskip("mpmath")


def pin_bruteforce(impl):
    """Explicit exp / sum at 50 digits on small rows, ragged lengths included."""
    mpmath.mp.dps = 50
    g = np.random.default_rng(11)
    for rows, T, scale in [(3, 1, 1.0), (2, 7, 3.0), (4, 13, 0.5), (1, 33, 10.0)]:
        x = g.normal(size=(rows, T)) * scale
        z, lse = impl.softmax_rows(x)
        for i in range(rows):
            ex = [mpmath.exp(mpmath.mpf(v)) for v in x[i]]
            tot = mpmath.fsum(ex)
            assert abs(float(mpmath.log(tot)) - lse[i]) <= 1e-13
            for j in range(T):
                assert abs(float(ex[j] / tot) - z[i, j]) <= 1e-15


def pin_closed_forms(impl):
    # constant row: 1/T and lse = c + log T
    x = np.full((3, 10), 2.5)
    z, lse = impl.softmax_rows(x)
    np.testing.assert_allclose(z, 0.1, atol=1e-16, rtol=0)
    np.testing.assert_allclose(lse, 2.5 + math.log(10), atol=1e-14, rtol=0)
    # one entry far above the rest: z -> one-hot
    x = np.zeros((2, 6))
    x[0, 3] = 800.0
    x[1, 0] = 800.0
    z, lse = impl.softmax_rows(x)
    np.testing.assert_allclose(z, np.eye(6)[[3, 0]], atol=1e-300, rtol=0)
    np.testing.assert_allclose(lse, 800.0, atol=1e-12, rtol=0)
    # -inf entries get exactly zero probability
    x = np.array([[0.0, -np.inf, math.log(3.0)]])
    z, lse = impl.softmax_rows(x)
    np.testing.assert_allclose(z, [[0.25, 0.0, 0.75]], atol=1e-16, rtol=0)
    np.testing.assert_allclose(lse, [math.log(4.0)], atol=1e-15, rtol=0)
    # two entries: the logistic function
    a, b = 1.7, -0.4
    z, _ = impl.softmax_rows(np.array([[a, b]]))
    np.testing.assert_allclose(z[0, 0], 1.0 / (1.0 + math.exp(b - a)), atol=1e-16, rtol=0)


def pin_invariants(impl):
    g = np.random.default_rng(12)
    x = g.normal(size=(5, 40)) * 4
    z, lse = impl.softmax_rows(x)
    assert (z >= 0).all()
    np.testing.assert_allclose(z.sum(axis=1), 1.0, atol=1e-14, rtol=0)
    # shift by a row constant: z unchanged, lse shifted (exactly representable shifts)
    c = np.array([3.0, -2.0, 1000.0, 0.5, -700.0])
    z2, lse2 = impl.softmax_rows(x + c[:, None])
    np.testing.assert_allclose(z2, z, atol=1e-13, rtol=0)
    np.testing.assert_allclose(lse2, lse + c, atol=1e-10, rtol=0)
    # permuting a row permutes z
    perm = g.permutation(40)
    z3, lse3 = impl.softmax_rows(x[:, perm])
    np.testing.assert_allclose(z3, z[:, perm], atol=1e-15, rtol=0)
    np.testing.assert_allclose(lse3, lse, atol=1e-13, rtol=0)
    # huge magnitudes stay finite (the max subtraction)
    big = np.array([[1.0e4, 1.0e4 - 1.0, 1.0e4 - 2.0]])
    zb, lb = impl.softmax_rows(big)
    e = np.exp([0.0, -1.0, -2.0])
    np.testing.assert_allclose(zb, [e / e.sum()], atol=1e-15, rtol=0)
    np.testing.assert_allclose(lb, [1.0e4 + math.log(e.sum())], atol=1e-10, rtol=0)


ALL_PINS = [pin_bruteforce, pin_closed_forms, pin_invariants]


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(pin):
    pin(ref)


def _no_max(x):
    x = np.asarray(x, float)
    with np.errstate(all="ignore"):
        e = np.exp(x)
        s = e.sum(axis=1)
        return e / s[:, None], np.log(s)


def _drops_tail(x):
    x = np.asarray(x, float)
    z, lse = ref.softmax_rows(x[:, :-1]) if x.shape[1] > 1 else ref.softmax_rows(x)
    if x.shape[1] > 1:
        z = np.concatenate([z, np.zeros((x.shape[0], 1))], axis=1)
    return z, lse


def _column_softmax(x):
    z, _ = ref.softmax_rows(np.asarray(x, float).T)
    _, lse = ref.softmax_rows(x)
    return z.T, lse


MUTANTS = {"no_max": _no_max, "drops_tail": _drops_tail, "column_softmax": _column_softmax}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    impl = types.SimpleNamespace(softmax_rows=MUTANTS[name])
    failures = 0
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(impl)
        except (AssertionError, ValueError, FloatingPointError, IndexError):
            failures += 1
    assert failures >= 1, f"planted mistake {name} passed every pin"
