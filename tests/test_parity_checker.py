"""The backward parity checker (tests/parity.py) accepts what a correct
kernel returns and rejects planted mistakes, on the CPU.

A correct result is stood in for by the float64 oracle's gradients rounded to
the input type (what a kernel without any error of its own would return) and
by the same-precision naive reference itself.  Each mistake is planted into a
copy of the rounded oracle gradients.  The mistakes include the one the
per-head bound alone cannot see: zeroing the rows whose gradients are small
next to the head's largest (in a long causal bf16 head a sizable share of
dV's rows lies wholly below 1e-2 x max |dV|).
"""

import numpy as np
import pytest
import torch

import oracle.attention as ref
from tiled_attention_07_gb300 import workloads as W

from parity import GRAD_TOL, check_grads, half_ulp, naive_grads, rounding_sigma

CASES = [
    # dtype, Nq, Nk, d, causal, std
    ("bf16", 1024, 1024, 80, True, 1.0),
    ("fp16", 300, 700, 64, False, 0.5),
    ("bf16", 640, 256, 128, True, 1.0),
]


def _setup(case):
    dtype, nq, nk, d, causal, std = case
    w = W.custom(dtype, "bhsd", 1, 1, nq, nk, d, causal, std=std, seed=nq + nk + d, backward=True)
    x = W.make_inputs(w)
    q, k, v, do = (x[n][0, 0].double().numpy() for n in ("q", "k", "v", "do"))
    dq, dk, dv, _ = ref.backward(q, k, v, do, w.sm_scale, w.causal)
    exact = {"dq": dq, "dk": dk, "dv": dv}
    naive = dict(zip(("dq", "dk", "dv"), naive_grads(q, k, v, do, w.sm_scale, w.causal, w.dtype)))
    sigma = dict(zip(("dq", "dk", "dv"), rounding_sigma(q, k, v, do, w.sm_scale, w.causal, w.dtype)))
    rounded = {n: torch.from_numpy(a).to(w.torch_dtype).double().numpy() for n, a in exact.items()}
    return w, exact, naive, rounded, sigma


def _round(a, dtype):
    return torch.from_numpy(a).to(W.DTYPES[dtype]).double().numpy()


def _per_head_bound_only(dtype, got, exact):
    """The per-head bound (a) on its own: True if it accepts `got`."""
    for n in ("dq", "dk", "dv"):
        r = exact[n]
        excess = (np.abs(got[n] - r) - half_ulp(r, dtype)) / max(1.0, float(np.abs(r).max()))
        if excess.max() > GRAD_TOL[dtype]:
            return False
    return True


@pytest.fixture(scope="module", params=CASES, ids=["-".join(map(str, c)) for c in CASES])
def setup(request):
    return _setup(request.param)


def test_correct_results_pass(setup):
    w, exact, naive, rounded, sigma = setup
    stats = {}
    check_grads(w.dtype, rounded, exact, naive, "rounded oracle", stats, sigma)
    check_grads(w.dtype, naive, exact, naive, "naive", stats, sigma)
    # the rounded exact result sits well inside both bounds
    assert max(stats[f"max_row_frac_{n}"] for n in ("dq", "dk", "dv")) < 0.5, stats
    assert max(stats[f"max_tile_frac_{n}"] for n in ("dq", "dk", "dv")) < 0.5, stats


def _rows_below_head_tolerance(dtype, a):
    """Rows whose every element lies below the per-head bound (a): zeroing
    them is invisible to that bound."""
    lim = GRAD_TOL[dtype] * max(1.0, float(np.abs(a).max()))
    rows = np.abs(a).max(axis=1) < lim
    return rows & (np.abs(a).max(axis=1) > 0)


def _mutants(w, g):
    """(name, mutated copy of g) pairs; g holds the rounded oracle gradients."""
    nk = g["dv"].shape[0]
    out = []
    m = {n: a.copy() for n, a in g.items()}
    m["dv"][nk // 2:] = 0.0
    out.append(("dV rows >= Nk/2 zeroed", m))
    m = {n: a.copy() for n, a in g.items()}
    t0 = min(128, nk - 1)
    m["dk"][t0:t0 + 128] = _round(m["dk"][t0:t0 + 128] * 1.01, w.dtype)
    out.append(("dK 1 % high on one key tile", m))
    below = _rows_below_head_tolerance(w.dtype, g["dv"])
    if below.any():   # rows that small occur in long causal heads
        m = {n: a.copy() for n, a in g.items()}
        m["dv"][below] = 0.0
        out.append(("the dV rows below the per-head tolerance zeroed", m))
    m = {n: a.copy() for n, a in g.items()}
    r = int(np.argmax(np.linalg.norm(m["dq"], axis=1)))
    c = int(np.argmax(np.abs(m["dq"][r])))
    m["dq"][r, c] = -m["dq"][r, c]
    out.append(("one dQ element with its sign flipped", m))
    m = {n: a.copy() for n, a in g.items()}
    m["dk"][[5, 6]] = m["dk"][[6, 5]]
    out.append(("two adjacent dK rows swapped", m))
    m = {n: a.copy() for n, a in g.items()}
    m["dq"] = _round(m["dq"] * 0.99, w.dtype)
    out.append(("dQ 1 % low everywhere", m))
    return out


def test_planted_mistakes_are_rejected(setup):
    w, exact, naive, rounded, sigma = setup
    for name, m in _mutants(w, rounded):
        with pytest.raises(AssertionError):
            check_grads(w.dtype, m, exact, naive, name, {}, sigma)


def test_small_rows_zeroed_pass_the_per_head_bound_alone():
    # Why the per-row bound exists: on a long causal bf16 head, a sizable
    # share of dV's rows lies wholly below the per-head tolerance, and zeroing
    # all of them stays inside that bound.
    w, exact, naive, rounded, sigma = _setup(("bf16", 2048, 2048, 80, True, 1.0))
    share = _rows_below_head_tolerance(w.dtype, rounded["dv"]).mean()
    assert share > 0.1, share
    name, m = _mutants(w, rounded)[2]
    assert name.startswith("the dV rows below")
    assert _per_head_bound_only(w.dtype, m, exact)
    with pytest.raises(AssertionError, match="dv row"):
        check_grads(w.dtype, m, exact, naive, name, {}, sigma)


def test_short_causal_rows_with_a_few_ulps_of_error_pass():
    # A correct kernel's error on a row that sums a handful of terms can be
    # several times the naive reference's (both are a few random roundings):
    # three half-ulps of error on each early dQ row must still pass.
    w, exact, naive, rounded, sigma = _setup(("bf16", 1024, 1024, 80, True, 1.0))
    m = {n: a.copy() for n, a in rounded.items()}
    rng = np.random.default_rng(0)
    for i in range(1, 8):
        row = exact["dq"][i]
        m["dq"][i] = row + 3 * half_ulp(row, w.dtype) * rng.choice([-1.0, 1.0], size=row.shape)
    check_grads(w.dtype, m, exact, naive, "early rows", {}, sigma)


def test_naive_reference_follows_the_definition():
    # Pinned apart from the GPU: in float64, without the roundings, the naive
    # steps give the oracle's gradients; its error at the storage precision is
    # of the order of the output rounding (a few 2^-9 per row in bf16).
    w, exact, naive, rounded, sigma = _setup(("bf16", 256, 384, 64, True, 1.0))
    for n in ("dq", "dk", "dv"):
        rel = np.linalg.norm(naive[n] - exact[n], axis=1) / np.maximum(np.linalg.norm(exact[n], axis=1), 1e-30)
        live = np.linalg.norm(exact[n], axis=1) > 1e-6
        assert np.median(rel[live]) < 4 * 2.0 ** -9, (n, np.median(rel[live]))
    nf = dict(zip(("dq", "dk", "dv"), naive_grads(*_f64_inputs(w), w.sm_scale, w.causal, "fp32")))
    for n in ("dq", "dk", "dv"):
        np.testing.assert_allclose(nf[n], exact[n], rtol=0, atol=1e-5 * max(1.0, np.abs(exact[n]).max()))


def _f64_inputs(w):
    x = W.make_inputs(w)
    return tuple(x[n][0, 0].double().numpy() for n in ("q", "k", "v", "do"))


def _tiled_style(q, k, v, do, sm_scale, causal, dtype):
    """dQ, dK, dV computed a second way at the same precision, with the
    forward's roundings where a tiled kernel takes them: p = exp(s - m)
    unnormalised (m the row max) rounded before the product with V, O divided
    by the row sum and rounded; D from that O; P and dS rounded before their
    products; results rounded.  Its roundings are draws independent of the
    naive reference's, as a GPU kernel's are."""
    tdt = W.DTYPES[dtype]
    qf, kf, vf, dof = (torch.from_numpy(a).float() for a in (q, k, v, do))
    s = (qf @ kf.T) * sm_scale
    if causal:
        s = s.masked_fill(torch.arange(s.shape[1])[None, :] > torch.arange(s.shape[0])[:, None], float("-inf"))
    m = s.max(dim=-1, keepdim=True).values
    pu = torch.exp(s - m)
    lsum = pu.sum(dim=-1, keepdim=True)
    o = ((pu.to(tdt).float() @ vf) / lsum).to(tdt).float()
    p = pu / lsum
    dsum = (o * dof).sum(dim=-1, keepdim=True)
    dv = (p.to(tdt).float().T @ dof).to(tdt)
    ds = (p * (dof @ vf.T - dsum)).to(tdt).float()
    return tuple(t.double().numpy() for t in ((sm_scale * (ds @ kf)).to(tdt), (sm_scale * (ds.T @ qf)).to(tdt), dv))


@pytest.mark.parametrize("case", CASES + [("bf16", 4096, 4096, 80, True, 1.0), ("bf16", 4096, 4096, 64, True, 1.0)],
                         ids=lambda c: "-".join(map(str, c)))
def test_a_second_same_precision_computation_passes(case):
    w, exact, naive, rounded, sigma = _setup(case)
    x = W.make_inputs(w)
    q, k, v, do = (x[n][0, 0].double().numpy() for n in ("q", "k", "v", "do"))
    got = dict(zip(("dq", "dk", "dv"), _tiled_style(q, k, v, do, w.sm_scale, w.causal, w.dtype)))
    stats = {}
    check_grads(w.dtype, got, exact, naive, "tiled style", stats, sigma)
    print(case, {k: round(v, 3) for k, v in stats.items() if "frac" in k})


def test_a_vanishing_gradient_with_rounding_noise_passes():
    # One query and one key: dQ is exactly zero and so is the naive
    # reference's error; a kernel's float32 noise there must pass, while a
    # real error does not.
    w, exact, naive, rounded, sigma = _setup(("bf16", 1, 1, 64, True, 1.0))
    assert np.all(exact["dq"] == 0) and np.all(naive["dq"] == 0)
    m = {n: a.copy() for n, a in rounded.items()}
    m["dq"][0, :4] = 6e-8
    check_grads(w.dtype, m, exact, naive, "noise", {}, sigma)
    m["dv"] = -m["dv"]
    with pytest.raises(AssertionError):
        check_grads(w.dtype, m, exact, naive, "sign", {}, sigma)
