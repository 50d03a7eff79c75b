"""Pins of the fp8 (e5m2) V oracle to the format's definition, to a library
conversion, to closed forms and to a hand-derived example.

What is pinned, and the mistake each pin is there to catch:
* the decoder against every code of torch's float8_e5m2 (a library routine)
  and against codes decoded by hand from the format's definition;
* the encoder against torch's round-to-nearest cast on random values of every
  binade, and against hand-worked ties (ties go to the even code);
* the forward: one key (O = v_0 exactly), equal scores (p = 1 is exact in
  e5m2, so O is the plain mean of the visible keys), a two-key example whose
  result is worked out by hand below, the bound |O - O_exact| <= 2^-3 max|v|
  that the cast allows, and the LSE, which takes unrounded p and so equals the
  exact one;
* planted mistakes (no cast, a 3-bit-mantissa cast, l over the cast p) fail
  the hand-derived example.
"""

import math
import types

import numpy as np
import pytest
import torch

import oracle.attention as exact
import oracle.fp8 as f8


# ---------------------------------------------------------------------------
# the format
# ---------------------------------------------------------------------------

def test_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = f8.e5m2_decode(codes)
    theirs = torch.from_numpy(codes).view(torch.float8_e5m2).to(torch.float64).numpy()
    finite = np.isfinite(theirs)
    assert np.array_equal(np.isfinite(ours), finite)
    assert np.array_equal(ours[finite], theirs[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(theirs))
    assert np.array_equal(ours[np.isinf(theirs)], theirs[np.isinf(theirs)])


@pytest.mark.parametrize("code,value", [
    (0x3C, 1.0),                 # e = 15, f = 0
    (0x38, 0.5),                 # e = 14
    (0x3D, 1.25),                # f = 1: 1 + 1/4
    (0x3E, 1.5),
    (0x3F, 1.75),
    (0x7B, 57344.0),             # e = 30, f = 3: 1.75 * 2^15
    (0x04, 2.0 ** -14),          # smallest normal
    (0x01, 2.0 ** -16),          # smallest subnormal
    (0x03, 3 * 2.0 ** -16),
    (0xBC, -1.0),
    (0x00, 0.0),
])
def test_decode_by_hand(code, value):
    assert f8.e5m2_decode(np.array([code], dtype=np.uint8))[0] == value


def test_decode_specials():
    assert f8.e5m2_decode(np.array([0x7C], dtype=np.uint8))[0] == np.inf
    assert f8.e5m2_decode(np.array([0xFC], dtype=np.uint8))[0] == -np.inf
    assert np.isnan(f8.e5m2_decode(np.array([0x7D], dtype=np.uint8))[0])


def test_encode_matches_torch_cast():
    g = np.random.default_rng(5)
    x = np.concatenate([
        g.standard_normal(4000) * np.exp2(g.uniform(-18, 15, 4000)),   # every binade, both signs
        g.uniform(0, 1, 2000),                                          # the range of p
        g.uniform(-2.0 ** -14, 2.0 ** -14, 1000),                       # subnormals
    ])
    x = x[np.abs(x) <= f8.E5M2_MAX]   # torch's cast overflows to inf beyond it; ours saturates (pinned by hand)
    ours = f8.e5m2_encode(x)
    theirs = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


@pytest.mark.parametrize("x,value", [
    (1.125, 1.0),                # halfway between 1.0 (f = 0) and 1.25 (f = 1): even f
    (1.375, 1.5),                # halfway between 1.25 (f = 1) and 1.5 (f = 2): even f
    (1.875, 2.0),                # halfway between 1.75 and 2.0: even (next binade, f = 0)
    (0.7, 0.75),                 # 1.4 * 2^-1: 1.5 is nearer than 1.25
    (0.6, 0.625),                # 1.2 * 2^-1: 1.25 is nearer than 1.0
    (2.0 ** -17, 0.0),           # half the smallest subnormal: tie to 0
    (3 * 2.0 ** -17, 2.0 ** -15),   # 1.5 subnormal units: tie to 2 units
    (60000.0, 57344.0),          # saturates
    (-0.7, -0.75),
])
def test_round_by_hand(x, value):
    assert f8.e5m2_round(np.array([x]))[0] == value


# ---------------------------------------------------------------------------
# the forward
# ---------------------------------------------------------------------------

def _inputs(g, nq, nk, d, std=1.0):
    q = g.standard_normal((nq, d)) * std
    k = g.standard_normal((nk, d)) * std
    vt = f8.e5m2_round(g.standard_normal((d, nk)))
    return q, k, vt


@pytest.mark.parametrize("causal", [False, True])
def test_one_key(causal):
    g = np.random.default_rng(1)
    q, k, vt = _inputs(g, 5, 1, 4)
    o, lse = f8.forward_fp8v(q, k, vt, 0.5, causal)
    assert np.array_equal(o, np.broadcast_to(vt[:, 0], o.shape))
    assert np.allclose(lse, 0.5 * (q @ k[0]), rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block_n", [3, 128])
def test_equal_scores_mean(causal, block_n):
    # Q = 0: every score is 0, every p is exactly 1 (also after the cast), so
    # O_i is the mean of the visible V rows and LSE_i = log(#visible).
    g = np.random.default_rng(2)
    nq, nk, d = 7, 9, 3
    q = np.zeros((nq, d))
    k = g.standard_normal((nk, d))
    vt = f8.e5m2_round(g.standard_normal((d, nk)))
    o, lse = f8.forward_fp8v(q, k, vt, 1.0, causal, block_n)
    for i in range(nq):
        n = min(i + 1, nk) if causal else nk
        assert np.allclose(o[i], vt[:, :n].mean(axis=1), rtol=0, atol=1e-14)
        assert abs(lse[i] - math.log(n)) < 1e-14


def _two_key_case():
    # d = 1, sm_scale = 1, q = 1: scores s_0 = 0 (the row max) and
    # s_1 = ln 0.7, so p_0 = 1 and p_1 = 0.7; V = (1, 2).  The cast turns p_1
    # into 0.75 (1.4 * 2^-1 rounds to 1.5 * 2^-1) while l keeps 1.7:
    #   O = (1 * 1 + 0.75 * 2) / 1.7 = 2.5 / 1.7
    # (the exact result is (1 + 0.7 * 2) / 1.7 = 2.4 / 1.7).
    q = np.array([[1.0]])
    k = np.array([[0.0], [math.log(0.7)]])
    vt = np.array([[1.0, 2.0]])
    return q, k, vt, 2.5 / 1.7, math.log(1.7)


def _check_two_key(impl):
    q, k, vt, o_ref, lse_ref = _two_key_case()
    o, lse = impl.forward_fp8v(q, k, vt, 1.0, False)
    assert abs(o[0, 0] - o_ref) < 1e-12 and abs(lse[0] - lse_ref) < 1e-12


def test_two_key_by_hand():
    _check_two_key(f8)


def test_lse_equals_exact_and_o_within_cast_bound():
    g = np.random.default_rng(3)
    for causal, (nq, nk, d), bn in [(False, (33, 70, 8), 16), (True, (40, 40, 16), 8), (True, (20, 50, 4), 128)]:
        q, k, vt = _inputs(g, nq, nk, d, std=1.5)
        o, lse = f8.forward_fp8v(q, k, vt, 0.4, causal, bn)
        o_ex, lse_ex = exact.forward(q, k, vt.T, 0.4, causal)
        assert np.allclose(lse, lse_ex, rtol=0, atol=1e-12)
        for i in range(nq):
            n = min(i + 1, nk) if causal else nk
            bound = 2.0 ** -3 * np.max(np.abs(vt[:, :n])) + 1e-12
            assert np.max(np.abs(o[i] - o_ex[i])) <= bound
        # and the cast does change O (the check above is not vacuous)
        assert np.max(np.abs(o - o_ex)) > 1e-6


# ---------------------------------------------------------------------------
# planted mistakes
# ---------------------------------------------------------------------------

def _mutant(round_fn=None, l_of_cast=False):
    def forward_fp8v(q, k, vt, sm_scale, causal, block_n=128):
        q = np.asarray(q, dtype=np.float64)
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(vt, dtype=np.float64).T
        c = sm_scale * math.log2(math.e)
        nq = q.shape[0]
        m = np.full(nq, -np.inf)
        l = np.zeros(nq)
        acc = np.zeros((nq, v.shape[1]))
        for j0 in range(0, k.shape[0], block_n):
            qk = q @ k[j0:j0 + block_n].T
            m_new = np.maximum(m, qk.max(axis=1) * c)
            p = np.exp2(qk * c - m_new[:, None])
            alpha = np.where(np.isfinite(m), np.exp2(m - m_new), 0.0)
            pr = round_fn(p)
            l = l * alpha + (pr if l_of_cast else p).sum(axis=1)
            acc = acc * alpha[:, None] + pr @ v[j0:j0 + block_n]
            m = m_new
        return acc / l[:, None], (m + np.log2(l)) * math.log(2.0)
    return types.SimpleNamespace(forward_fp8v=forward_fp8v)


def _e4m3_round(p):   # 3 mantissa bits, normal range only (enough for p in (2^-6, 1])
    e = np.floor(np.log2(p))
    return np.round(p / 2.0 ** (e - 3)) * 2.0 ** (e - 3)


@pytest.mark.parametrize("mutant", [
    _mutant(round_fn=lambda p: p),                       # no cast
    _mutant(round_fn=_e4m3_round),                       # the other float8 format
    _mutant(round_fn=f8.e5m2_round, l_of_cast=True),     # l over the cast p
])
def test_pins_catch_mistakes(mutant):
    with pytest.raises(AssertionError):
        _check_two_key(mutant)
