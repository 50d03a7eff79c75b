"""Pins of the float64 oracle to facts the pages and the mathematics fix.

Each check is written against an *implementation object* (anything with
``probabilities``, ``forward`` and ``backward`` like ``oracle.attention``), so
the same checks also run against planted mistakes (see ``test_pins_catch_*``):
a plausible bug in the oracle (a dropped term, a wrong sign or index, a
transposed operand) must fail at least one pin.

Pins:
* brute force at 50 significant digits (mpmath) on tiny inputs, including
  causal and Nq != Nk;
* hand-derived worked examples (tests/golden/closed_form_cases.json);
* closed forms: Nk = 1, constant V, Q = 0, one dominating score;
* invariants: softmax rows sum to 1, shift of all scores, causal masking
  invariance, key permutation, query permutation;
* backward: central finite differences of sum(O * dO), the identity
  rowsum(P o dP) = rowsum(O o dO), and sum_j dK_j = 0.
"""

import json
import math
import os
import types

import numpy as np
import pytest

import oracle.attention as ref

mpmath = pytest.importorskip("mpmath")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")


def rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# pins as functions of an implementation
# ---------------------------------------------------------------------------

def pin_bruteforce(impl):
    """Explicit softmax at 50 digits: O_i = sum_j e^{s_ij} v_j / sum_j e^{s_ij}."""
    mpmath.mp.dps = 50
    g = rng(1)
    for (nq, nk, d, causal, scale) in [(3, 5, 2, False, 0.7), (5, 3, 3, True, 1.3), (4, 4, 1, True, 0.5),
                                       (2, 6, 4, False, 2.0), (6, 2, 2, True, 0.9)]:
        q = g.normal(size=(nq, d))
        k = g.normal(size=(nk, d))
        v = g.normal(size=(nk, d))
        o, lse = impl.forward(q, k, v, scale, causal)
        for i in range(nq):
            ex = []
            for j in range(nk):
                if causal and j > i:
                    continue
                s = mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[i, t]) * mpmath.mpf(k[j, t]) for t in range(d))
                ex.append((j, mpmath.exp(s)))
            z = mpmath.fsum(e for _, e in ex)
            assert abs(float(mpmath.log(z)) - lse[i]) <= 1e-12, "lse"
            for t in range(d):
                oi = mpmath.fsum(e * mpmath.mpf(v[j, t]) for j, e in ex) / z
                assert abs(float(oi) - o[i, t]) <= 1e-12, "O"


def _num(x):
    if isinstance(x, str):
        x = x.replace("ln", "math.log")
        x = x.replace("math.log3", "math.log(3)").replace("math.log4", "math.log(4)")
        return float(eval(x, {"math": math}))
    return float(x)


def _arr(rows):
    return np.array([[_num(x) for x in r] for r in rows], dtype=np.float64)


def pin_golden(impl):
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q, k, v, do = _arr(c["q"]), _arr(c["k"]), _arr(c["v"]), _arr(c["do"])
        o, lse = impl.forward(q, k, v, c["sm_scale"], c["causal"])
        np.testing.assert_allclose(o, _arr(c["o"]), atol=1e-14, rtol=0, err_msg=c["name"])
        np.testing.assert_allclose(lse, [_num(x) for x in c["lse"]], atol=1e-14, rtol=0, err_msg=c["name"])
        dq, dk, dv, _ = impl.backward(q, k, v, do, c["sm_scale"], c["causal"])
        np.testing.assert_allclose(dq, _arr(c["dq"]), atol=1e-14, rtol=0, err_msg=c["name"])
        np.testing.assert_allclose(dk, _arr(c["dk"]), atol=1e-14, rtol=0, err_msg=c["name"])
        np.testing.assert_allclose(dv, _arr(c["dv"]), atol=1e-14, rtol=0, err_msg=c["name"])


def pin_closed_forms(impl):
    g = rng(2)
    # Nk = 1: O = V_0, LSE = S_00
    q = g.normal(size=(7, 5))
    k = g.normal(size=(1, 5))
    v = g.normal(size=(1, 5))
    for causal in (False, True):
        o, lse = impl.forward(q, k, v, 0.8, causal)
        np.testing.assert_allclose(o, np.repeat(v, 7, axis=0), atol=1e-14, rtol=0)
        np.testing.assert_allclose(lse, 0.8 * (q @ k[0]), atol=1e-13, rtol=0)
    # constant V -> constant O
    q = g.normal(size=(6, 4))
    k = g.normal(size=(9, 4))
    v = np.tile(np.array([[1.5, -2.0, 0.25, 3.0]]), (9, 1))
    for causal in (False, True):
        o, _ = impl.forward(q, k, v, 1.1, causal)
        np.testing.assert_allclose(o, np.tile(v[:1], (6, 1)), atol=1e-13, rtol=0)
    # Q = 0 -> O = mean of the visible V rows, LSE = log(#visible)
    nq, nk = 5, 8
    q = np.zeros((nq, 3))
    k = g.normal(size=(nk, 3))
    v = g.normal(size=(nk, 3))
    o, lse = impl.forward(q, k, v, 0.5, False)
    np.testing.assert_allclose(o, np.tile(v.mean(axis=0), (nq, 1)), atol=1e-14, rtol=0)
    np.testing.assert_allclose(lse, np.full(nq, math.log(nk)), atol=1e-14, rtol=0)
    o, lse = impl.forward(q, k, v, 0.5, True)
    for i in range(nq):
        np.testing.assert_allclose(o[i], v[: i + 1].mean(axis=0), atol=1e-14, rtol=0)
        assert abs(lse[i] - math.log(i + 1)) <= 1e-14
    # one dominating score: O -> V_argmax
    q = np.array([[1.0, 0.0]])
    k = np.array([[0.0, 1.0], [60.0, 0.0], [-3.0, 2.0]])
    v = g.normal(size=(3, 2))
    o, lse = impl.forward(q, k, v, 1.0, False)
    np.testing.assert_allclose(o[0], v[1], atol=1e-20 + 1e-24, rtol=1e-20)
    assert abs(lse[0] - 60.0) <= 1e-20 + 1e-24


def pin_invariants(impl):
    g = rng(3)
    nq, nk, d = 9, 13, 6
    q = g.normal(size=(nq, d))
    k = g.normal(size=(nk, d))
    v = g.normal(size=(nk, d))
    for causal in (False, True):
        p, lse = impl.probabilities(q, k, 0.6, causal)
        assert p.shape == (nq, nk)
        assert np.all(p >= 0)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12, rtol=0)
        if causal:
            i = np.arange(nq)[:, None]
            j = np.arange(nk)[None, :]
            assert np.all(p[j > i] == 0.0)
            assert np.all(p[j <= i] > 0.0)
        # shift: an extra coordinate adds a to every score of every row
        a = 2.75
        scale = 0.6
        q2 = np.concatenate([q, np.ones((nq, 1))], axis=1)
        k2 = np.concatenate([k, np.full((nk, 1), a / scale)], axis=1)
        p2, lse2 = impl.probabilities(q2, k2, scale, causal)
        np.testing.assert_allclose(p2, p, atol=1e-13, rtol=0)
        np.testing.assert_allclose(lse2, lse + a, atol=1e-12, rtol=0)
    # causal masking invariance: keys after row i do not change row i at all
    o, lse = impl.forward(q, k, v, 0.6, True)
    for i in range(nq):
        k2 = k.copy()
        v2 = v.copy()
        k2[i + 1:] = g.normal(size=k2[i + 1:].shape) * 10
        v2[i + 1:] = g.normal(size=v2[i + 1:].shape) * 10
        o2, lse2 = impl.forward(q, k2, v2, 0.6, True)
        assert np.array_equal(o2[i], o[i])
        assert lse2[i] == lse[i]
    # key permutation (K and V together) leaves the non-causal result unchanged
    o, lse = impl.forward(q, k, v, 0.6, False)
    perm = g.permutation(nk)
    o2, lse2 = impl.forward(q, k[perm], v[perm], 0.6, False)
    np.testing.assert_allclose(o2, o, atol=1e-13, rtol=0)
    np.testing.assert_allclose(lse2, lse, atol=1e-13, rtol=0)
    # query permutation permutes the rows
    perm = g.permutation(nq)
    o2, lse2 = impl.forward(q[perm], k, v, 0.6, False)
    np.testing.assert_allclose(o2, o[perm], atol=1e-13, rtol=0)
    np.testing.assert_allclose(lse2, lse[perm], atol=1e-13, rtol=0)


def pin_finite_differences(impl):
    """Central differences of loss = sum(O * dO) against the analytic backward."""
    g = rng(4)
    h = 1e-6
    for (nq, nk, d, causal, scale) in [(4, 6, 3, False, 0.7), (5, 5, 2, True, 1.2), (6, 3, 3, True, 0.5)]:
        q = g.normal(size=(nq, d))
        k = g.normal(size=(nk, d))
        v = g.normal(size=(nk, d))
        do = g.normal(size=(nq, d))
        dq, dk, dv, _ = impl.backward(q, k, v, do, scale, causal)

        def loss(q_, k_, v_):
            o, _ = impl.forward(q_, k_, v_, scale, causal)
            return float(np.sum(o * do))

        for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp = x.copy()
                xm = x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = {"q": q, "k": k, "v": v}
                args_m = {"q": q, "k": k, "v": v}
                args_p[name] = xp
                args_m[name] = xm
                num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"]) - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
            err = np.max(np.abs(num - grad)) / max(1.0, np.max(np.abs(num)))
            assert err <= 1e-6, (name, causal, err)


def pin_backward_identities(impl):
    g = rng(5)
    nq, nk, d = 8, 11, 5
    q = g.normal(size=(nq, d))
    k = g.normal(size=(nk, d))
    v = g.normal(size=(nk, d))
    do = g.normal(size=(nq, d))
    for causal in (False, True):
        o, _ = impl.forward(q, k, v, 0.9, causal)
        dq, dk, dv, dsum = impl.backward(q, k, v, do, 0.9, causal)
        # D = rowsum(P o dP) = rowsum(O o dO)
        np.testing.assert_allclose(dsum, np.sum(o * do, axis=1), atol=1e-12, rtol=0)
        # rows of dS sum to zero, so sum_j dK_j = sm_scale * (sum_j dS_j)^T Q = 0
        np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12, rtol=0)
        # dV columns sum to dO columns because P rows sum to 1
        np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), atol=1e-12, rtol=0)


def pin_split_merge(impl):
    """Softmaxes over disjoint key ranges, merged, equal the softmax over all keys.

    Checked against the full forward (itself pinned by brute force above):
    random partitions of the keys, with empty ranges and ranges a causal row
    sees none of, and the one-range partition."""
    g = rng(7)
    for (nq, nk, d, causal, scale) in [(9, 13, 3, False, 0.8), (11, 11, 4, True, 1.2), (6, 15, 2, True, 0.6),
                                       (14, 5, 3, True, 1.5), (7, 20, 5, False, 2.5)]:
        q = g.normal(size=(nq, d))
        k = g.normal(size=(nk, d))
        v = g.normal(size=(nk, d))
        o_ref, lse_ref = impl.forward(q, k, v, scale, causal)
        o1, lse1 = impl.forward_keys(q, k, v, scale, causal, 0, nk)
        np.testing.assert_allclose(o1, o_ref, atol=1e-13, rtol=0)
        np.testing.assert_allclose(lse1, lse_ref, atol=1e-13, rtol=0)
        for trial in range(4):
            cuts = np.sort(g.integers(0, nk + 1, size=g.integers(1, 5)))
            bounds = [0] + list(cuts) + [nk]
            parts = [impl.forward_keys(q, k, v, scale, causal, a, b) for a, b in zip(bounds[:-1], bounds[1:])]
            o, lse = impl.merge([p[0] for p in parts], [p[1] for p in parts])
            np.testing.assert_allclose(o, o_ref, atol=1e-13, rtol=0)
            np.testing.assert_allclose(lse, lse_ref, atol=1e-13, rtol=0)


ALL_PINS = [pin_bruteforce, pin_golden, pin_closed_forms, pin_invariants, pin_finite_differences,
            pin_backward_identities, pin_split_merge]


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(pin):
    pin(ref)


def test_batched_helpers_match_single_head():
    g = rng(6)
    B, H, nq, nk, d = 2, 3, 5, 7, 4
    q = g.normal(size=(B, H, nq, d))
    k = g.normal(size=(B, H, nk, d))
    v = g.normal(size=(B, H, nk, d))
    do = g.normal(size=(B, H, nq, d))
    o, lse = ref.forward_heads(q, k, v, 0.4, True)
    dq, dk, dv = ref.backward_heads(q, k, v, do, 0.4, True)
    for b in range(B):
        for h in range(H):
            o1, l1 = ref.forward(q[b, h], k[b, h], v[b, h], 0.4, True)
            assert np.array_equal(o[b, h], o1) and np.array_equal(lse[b, h], l1)
            g1 = ref.backward(q[b, h], k[b, h], v[b, h], do[b, h], 0.4, True)
            assert np.array_equal(dq[b, h], g1[0]) and np.array_equal(dk[b, h], g1[1])
            assert np.array_equal(dv[b, h], g1[2])
    o, _ = ref.forward_heads(q, k, v, 0.4, False, heads=[(1, 2)])
    assert np.isnan(o[0, 0]).all() and not np.isnan(o[1, 2]).any()


# ---------------------------------------------------------------------------
# planted mistakes: each must be caught by at least one pin
# ---------------------------------------------------------------------------

def _mutant(scores=None, probabilities=None, forward=None, backward=None, forward_keys=None, merge=None):
    """An implementation object built from the oracle with one piece replaced."""
    m = types.SimpleNamespace()
    m.scores = scores or ref.scores

    def _probs(q, k, sm_scale, causal):
        s = m.scores(q, k, sm_scale, causal)
        mx = np.max(s, axis=1)
        lse = mx + np.log(np.sum(np.exp(s - mx[:, None]), axis=1))
        return np.exp(s - lse[:, None]), lse

    m.probabilities = probabilities or _probs

    def _fwd(q, k, v, sm_scale, causal):
        p, lse = m.probabilities(q, k, sm_scale, causal)
        return p @ np.asarray(v, float), lse

    m.forward = forward or _fwd

    def _bwd(q, k, v, do, sm_scale, causal):
        p, _ = m.probabilities(q, k, sm_scale, causal)
        dv = p.T @ do
        dp = do @ np.asarray(v, float).T
        dsum = np.sum(p * dp, axis=1)
        ds = p * (dp - dsum[:, None])
        return sm_scale * ds @ k, sm_scale * ds.T @ q, dv, dsum

    m.backward = backward or _bwd
    m.forward_keys = forward_keys or ref.forward_keys
    m.merge = merge or ref.merge
    return m


def _scores_no_scale(q, k, sm_scale, causal):
    return ref.scores(q, k, 1.0, causal)


def _scores_mask_flipped(q, k, sm_scale, causal):
    s = sm_scale * (np.asarray(q, float) @ np.asarray(k, float).T)
    if causal:
        i = np.arange(s.shape[0])[:, None]
        j = np.arange(s.shape[1])[None, :]
        s = np.where(j < i, -np.inf, s)
    return s


def _scores_mask_off_by_one(q, k, sm_scale, causal):
    s = sm_scale * (np.asarray(q, float) @ np.asarray(k, float).T)
    if causal:
        i = np.arange(s.shape[0])[:, None]
        j = np.arange(s.shape[1])[None, :]
        s = np.where(j >= i + 1 + 1, -np.inf, s)
    return s


def _probs_lse_missing_max(q, k, sm_scale, causal):
    s = ref.scores(q, k, sm_scale, causal)
    mx = np.max(s, axis=1)
    lse_wrong = np.log(np.sum(np.exp(s - mx[:, None]), axis=1))
    p = np.exp(s - mx[:, None]) / np.sum(np.exp(s - mx[:, None]), axis=1)[:, None]
    return p, lse_wrong


def _probs_column_softmax(q, k, sm_scale, causal):
    s = ref.scores(q, k, sm_scale, causal)
    e = np.exp(s - np.max(s))
    col = e.sum(axis=0)
    col[col == 0] = 1.0
    p = e / col[None, :]
    lse = np.log(np.sum(np.exp(s), axis=1))
    return p, lse


def _bwd_dropped_d(q, k, v, do, sm_scale, causal):
    p, _ = ref.probabilities(q, k, sm_scale, causal)
    dp = do @ np.asarray(v, float).T
    ds = p * dp
    return sm_scale * ds @ k, sm_scale * ds.T @ q, p.T @ do, np.sum(p * dp, axis=1)


def _bwd_dq_unscaled(q, k, v, do, sm_scale, causal):
    dq, dk, dv, dsum = ref.backward(q, k, v, do, sm_scale, causal)
    return dq / sm_scale, dk, dv, dsum


def _bwd_dk_wrong_operand(q, k, v, do, sm_scale, causal):
    p, _ = ref.probabilities(q, k, sm_scale, causal)
    dp = do @ np.asarray(v, float).T
    dsum = np.sum(p * dp, axis=1)
    ds = p * (dp - dsum[:, None])
    dk = sm_scale * (p.T @ q)  # P instead of dS
    return sm_scale * ds @ k, dk, p.T @ do, dsum


def _bwd_dv_untransposed(q, k, v, do, sm_scale, causal):
    dq, dk, dv, dsum = ref.backward(q, k, v, do, sm_scale, causal)
    p, _ = ref.probabilities(q, k, sm_scale, causal)
    if p.shape[0] == p.shape[1]:
        dv = p @ do
    else:
        dv = dv[::-1].copy()
    return dq, dk, dv, dsum


def _bwd_sign_flip(q, k, v, do, sm_scale, causal):
    dq, dk, dv, dsum = ref.backward(q, k, v, do, sm_scale, causal)
    return -dq, dk, dv, dsum


def _merge_equal_weights(o_parts, lse_parts):
    o_parts = np.asarray(o_parts, float)
    lse_parts = np.asarray(lse_parts, float)
    seen = np.isfinite(lse_parts)
    o = np.sum(np.where(seen[..., None], o_parts, 0.0), axis=0) / np.maximum(seen.sum(axis=0), 1)[:, None]
    return o, ref.merge(o_parts, lse_parts)[1]


def _forward_keys_relative_mask(q, k, v, sm_scale, causal, k_begin, k_end):
    # causal mask applied with key indices relative to the range
    return ref.forward_keys(q, np.asarray(k, float)[k_begin:k_end], np.asarray(v, float)[k_begin:k_end],
                            sm_scale, causal, 0, k_end - k_begin)


MUTANTS = {
    "no_scale": _mutant(scores=_scores_no_scale),
    "mask_flipped": _mutant(scores=_scores_mask_flipped),
    "mask_off_by_one": _mutant(scores=_scores_mask_off_by_one),
    "lse_missing_max": _mutant(probabilities=_probs_lse_missing_max),
    "column_softmax": _mutant(probabilities=_probs_column_softmax),
    "bwd_dropped_D": _mutant(backward=_bwd_dropped_d),
    "bwd_dq_unscaled": _mutant(backward=_bwd_dq_unscaled),
    "bwd_dk_wrong_operand": _mutant(backward=_bwd_dk_wrong_operand),
    "bwd_dv_untransposed": _mutant(backward=_bwd_dv_untransposed),
    "bwd_sign_flip": _mutant(backward=_bwd_sign_flip),
    "merge_equal_weights": _mutant(merge=_merge_equal_weights),
    "split_relative_mask": _mutant(forward_keys=_forward_keys_relative_mask),
}


def test_unmutated_rebuild_passes_every_pin():
    clean = _mutant()
    for pin in ALL_PINS:
        pin(clean)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    impl = MUTANTS[name]
    failures = 0
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(impl)
        except (AssertionError, ValueError, FloatingPointError, IndexError):
            failures += 1
    assert failures >= 1, f"planted mistake {name} passed every pin"
