"""Float64 CPU oracle for exact attention (forward, log-sum-exp, backward).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline
leg call it.  It shares no code with the CUDA library.

FlashAttention is exact: tiling and recomputation reorder the arithmetic but
reach the plain attention result ("[CS336] Assignment 2: Systems", section
"FlashAttention V2 / High level": the three techniques, and the statement
that the online logsumexp must equal the direct one).  So this oracle is the
plain definition, one (batch, head) matrix at a time, with S and P
materialised and every step in float64.

Definitions followed (all from "[CS336] Assignment 2: Systems", section
"FlashAttention V2 / High level"):

* forward:  S = sm_scale * Q K^T,  P_ij = softmax_j(S)_ij,  O = P V
* logsumexp: L_i = log sum_j exp(S_ij)
* backward:  dV = P^T dO,  dP = dO V^T,
             dS_i = (diag(P_i) - P_i P_i^T) dP_i,
             dQ = sm_scale * dS K,  dK = sm_scale * dS^T Q
* the identity rowsum(P o dP) = rowsum(O o dO) = D used by the recompute
  backward (same section, "D = rowsum(O o dO)").

Readings taken where the pages are open:

* ``sm_scale`` is a free parameter (the pages use both 1/sqrt(d) and 0.5).
* causal mask is top-left aligned: key j is visible to query i iff j <= i,
  also when Nq != Nk ("Understanding Triton Tutorials Part 2", "Fused
  Attention 2": the ``tril`` reference mask; "[CS336]" flash_fwd_kernel:
  ``q_idx < k_idx -> -inf``).  Masked entries have exactly zero probability.
* the log-sum-exp is the natural log of the scaled scores, per query row.

Parity: pinned (see tests/test_oracle.py): brute force at 50 digits on tiny
inputs, closed forms, invariants, finite differences of the backward.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "scores",
    "probabilities",
    "forward",
    "backward",
    "forward_keys",
    "merge",
    "forward_heads",
    "backward_heads",
]


def _as64(x) -> np.ndarray:
    a = np.asarray(x, dtype=np.float64)
    if a.ndim != 2:
        raise ValueError("expected a [seq, d] matrix")
    return a


def scores(q, k, sm_scale: float, causal: bool) -> np.ndarray:
    """S = sm_scale * Q K^T with masked entries set to -inf.

    "[CS336] Assignment 2: Systems", "FlashAttention V2 / High level", the
    definition S = QK^T / sqrt(d) with the scale left free; the causal mask
    keeps key j for query i iff j <= i (top-left).
    """
    q = _as64(q)
    k = _as64(k)
    s = float(sm_scale) * (q @ k.T)
    if causal:
        nq, nk = s.shape
        i = np.arange(nq)[:, None]
        j = np.arange(nk)[None, :]
        s = np.where(j > i, -np.inf, s)
    return s


def probabilities(q, k, sm_scale: float, causal: bool):
    """Row softmax P of S, and the row log-sum-exp L (natural log).

    L_i = log sum_j exp(S_ij) ("[CS336]", "FlashAttention V2 / High level",
    recomputation paragraph), evaluated stably as M_i + log sum_j
    exp(S_ij - M_i) with M_i the row maximum; P_ij = exp(S_ij - L_i), which is
    softmax_j(S)_ij.  Exp of -inf is exactly 0, so masked keys get P = 0.
    """
    s = scores(q, k, sm_scale, causal)
    m = np.max(s, axis=1)
    lse = m + np.log(np.sum(np.exp(s - m[:, None]), axis=1))
    p = np.exp(s - lse[:, None])
    return p, lse


def forward(q, k, v, sm_scale: float, causal: bool):
    """O = P V and the row log-sum-exp, for one (batch, head).

    Inputs are ``[Nq, d]``, ``[Nk, d]``, ``[Nk, d]``; returns ``(O [Nq, d],
    lse [Nq])`` in float64.
    """
    p, lse = probabilities(q, k, sm_scale, causal)
    o = p @ _as64(v)
    return o, lse


def forward_keys(q, k, v, sm_scale: float, causal: bool, k_begin: int, k_end: int):
    """The softmax of each query row over the keys [k_begin, k_end) only.

    Key indices are absolute (the causal mask still keeps key j for query i
    iff j <= i).  Returns ``(O_s [Nq, d], lse_s [Nq])``: O_s is P_s V with P_s
    the row softmax restricted to the range, lse_s the natural log of
    sum_{j in range} exp(S_ij).  A row that sees no key of the range has
    lse_s = -inf and O_s = 0 (an empty sum).
    """
    s = scores(q, k, sm_scale, causal)[:, k_begin:k_end]
    v = _as64(v)[k_begin:k_end]
    nq = s.shape[0]
    o = np.zeros((nq, v.shape[1]))
    lse = np.full(nq, -np.inf)
    for i in range(nq):
        row = s[i]
        if row.size == 0 or not np.isfinite(row).any():
            continue
        m = np.max(row)
        e = np.exp(row - m)
        z = np.sum(e)
        lse[i] = m + np.log(z)
        o[i] = (e / z) @ v
    return o, lse


def merge(o_parts, lse_parts):
    """Combine per-key-range softmax results into the softmax over their union.

    The rescaling step of the online softmax ("[CS336] Assignment 2:
    Systems", "FlashAttention V2 / Forward Pass": a new running max m' and
    l' = e^(m - m') l + ...; "Puzzles 8 Long Softmax": sum' = sum * exp(m1 -
    m2) + ...) applied to whole ranges: lse = log sum_s exp(lse_s) and
    O = sum_s exp(lse_s - lse) O_s.  ``o_parts`` is [S, Nq, d], ``lse_parts``
    [S, Nq]; ranges that a row does not see carry lse_s = -inf.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = np.max(lse_parts, axis=0)
    seen = np.isfinite(m)
    ms = np.where(seen, m, 0.0)
    w = np.exp(lse_parts - ms[None, :])                  # [S, Nq]; 0 for unseen ranges
    z = np.sum(w, axis=0)
    lse = np.where(seen, ms + np.log(np.where(seen, z, 1.0)), -np.inf)
    o = np.einsum("sn,snd->nd", w, o_parts) / np.where(seen, z, 1.0)[:, None]
    return o, lse


def backward(q, k, v, do, sm_scale: float, causal: bool):
    """dQ, dK, dV of loss = sum(O * dO) for one (batch, head), plus D.

    "[CS336] Assignment 2: Systems", "FlashAttention V2 / High level", the
    standard backward: dV = P^T dO, dP = dO V^T, dS_i = (diag(P_i) -
    P_i P_i^T) dP_i, dQ = sm_scale dS K, dK = sm_scale dS^T Q.  The softmax
    Jacobian-vector product is written out row-wise: (diag(p) - p p^T) g =
    p o g - p (p . g), i.e. dS = P o (dP - D) with D_i = sum_j P_ij dP_ij.

    Returns ``(dQ, dK, dV, D)`` in float64.
    """
    q = _as64(q)
    k = _as64(k)
    v = _as64(v)
    do = _as64(do)
    p, _ = probabilities(q, k, sm_scale, causal)
    dv = p.T @ do
    dp = do @ v.T
    dsum = np.sum(p * dp, axis=1)
    ds = p * dp - p * dsum[:, None]
    dq = float(sm_scale) * (ds @ k)
    dk = float(sm_scale) * (ds.T @ q)
    return dq, dk, dv, dsum


# ---------------------------------------------------------------------------
# batched helpers over [B, H, seq, d] float64 arrays
# ---------------------------------------------------------------------------

def forward_heads(q, k, v, sm_scale: float, causal: bool, heads=None):
    """Forward over ``[B, H, seq, d]`` arrays, head by head.

    ``heads`` optionally restricts the work to a list of (b, h) pairs; the
    other entries of the outputs are left as NaN.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, nq, d = q.shape
    o = np.full((B, H, nq, d), np.nan)
    lse = np.full((B, H, nq), np.nan)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    for b, h in heads:
        o[b, h], lse[b, h] = forward(q[b, h], k[b, h], v[b, h], sm_scale, causal)
    return o, lse


def backward_heads(q, k, v, do, sm_scale: float, causal: bool, heads=None):
    """Backward over ``[B, H, seq, d]`` arrays, head by head (see forward_heads)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, H, nq, d = q.shape
    nk = k.shape[2]
    dq = np.full((B, H, nq, d), np.nan)
    dk = np.full((B, H, nk, d), np.nan)
    dv = np.full((B, H, nk, d), np.nan)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    for b, h in heads:
        dq[b, h], dk[b, h], dv[b, h], _ = backward(q[b, h], k[b, h], v[b, h], do[b, h], sm_scale, causal)
    return dq, dk, dv
