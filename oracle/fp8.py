"""Float64 CPU oracle for the forward with V in float8 e5m2.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline
leg call it.  It shares no code with the CUDA library.

What the path computes ("Understanding Triton Tutorials Part 2", "Fused
Attention 2"): V is held in float8 e5m2 and stored transposed (its last two
dimensions are head dim, keys); in the inner loop of the forward the
probabilities p of a key block are cast to float8 e5m2 before the product
with V, while the row sum l takes the unrounded p.  The rest is that page's
online softmax, per key block of ``block_n`` keys:

    m_new = max(m, rowmax(qk) * c)          c = sm_scale * log2(e)
    p     = exp2(qk * c - m_new)
    alpha = exp2(m - m_new)
    l     = l * alpha + rowsum(p)
    acc   = acc * alpha + e5m2(p) V_block
    m     = m_new

and finally O = acc / l, LSE = ln 2 * (m + log2 l) (natural log of the
scaled scores, as the exact path).  The cast makes this an approximation
that depends on the blocks, so the oracle takes those steps in that order,
every step in float64 apart from the cast.

e5m2 (the float8 format with 5 exponent and 2 mantissa bits): sign bit,
exponent field e (bias 15), mantissa field f.  e = 0 gives subnormals
f * 2^-16; 1 <= e <= 30 gives (1 + f / 4) * 2^(e - 15), the largest finite
value being 1.75 * 2^15 = 57344; e = 31 is infinity (f = 0) or NaN.
Encoding rounds to nearest, ties to even; finite values beyond 57344
saturate to +-57344 (the conversion the GPU path uses saturates).

Parity: pinned (see tests/test_oracle_fp8.py): the decoder against every
code of torch's float8_e5m2 and hand-decoded codes, the rounding against
torch's cast and hand-worked ties, closed forms of the forward (one key;
equal scores), a hand-derived two-key example, and the cast bound
|O - O_exact| <= 2^-3 * max |v| per row.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = ["E5M2_MAX", "e5m2_decode", "e5m2_encode", "e5m2_round", "forward_fp8v", "forward_fp8v_heads"]

E5M2_MAX = 57344.0


def e5m2_decode(bits) -> np.ndarray:
    """Values (float64) of e5m2 codes given as unsigned 8-bit integers."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 2) & 0x1F
    f = (b & 0x3).astype(np.float64)
    sub = f * 2.0 ** -16
    nrm = (1.0 + f / 4.0) * np.exp2(e.astype(np.float64) - 15.0)
    special = np.where(f == 0, np.inf, np.nan)
    val = np.where(e == 0, sub, np.where(e == 31, special, nrm))
    return sign * val


def e5m2_encode(x) -> np.ndarray:
    """e5m2 codes of float64 values: round to nearest, ties to even, finite
    values beyond the largest finite one saturated; NaN -> 0x7F, +-inf ->
    0x7C / 0xFC."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint8)
    flat_x = x.reshape(-1)
    flat_o = out.reshape(-1)
    for i, v in enumerate(flat_x):
        flat_o[i] = _encode_one(float(v))
    return out


def _encode_one(v: float) -> int:
    if math.isnan(v):
        return 0x7F
    s = 0x80 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    if math.isinf(a):
        return s | 0x7C
    if a >= E5M2_MAX:
        return s | 0x7B
    # Units of the spacing of a's binade: subnormal spacing 2^-16 below
    # 2^-14, else 2^(E - 2) for a in [2^E, 2^(E+1)).
    if a < 2.0 ** -14:
        q = _round_half_even(a / 2.0 ** -16)    # 0 .. 4 (4 = smallest normal)
        return s | int(q)                       # code = mantissa units, e = 0 (or 1 when q = 4)
    E = math.floor(math.log2(a))
    if 2.0 ** E > a:                            # guard log2 rounding
        E -= 1
    elif 2.0 ** (E + 1) <= a:
        E += 1
    q = _round_half_even(a / 2.0 ** (E - 2))     # 4 .. 8
    if q == 8:
        E += 1
        q = 4
    if E > 15:                                  # rounded past 57344: saturate
        return s | 0x7B
    return s | ((E + 15) << 2) | (int(q) - 4)


def _round_half_even(t: float) -> int:
    fl = math.floor(t)
    r = t - fl
    if r > 0.5:
        return fl + 1
    if r < 0.5:
        return fl
    return fl if fl % 2 == 0 else fl + 1


def e5m2_round(x) -> np.ndarray:
    """x rounded to the nearest e5m2 value (ties to even, saturating)."""
    return e5m2_decode(e5m2_encode(x))


def forward_fp8v(q, k, vt, sm_scale: float, causal: bool, block_n: int = 128):
    """O and LSE of one (batch, head) with V in e5m2 and P cast to e5m2.

    ``q`` [Nq, d] and ``k`` [Nk, d] (float values), ``vt`` [d, Nk] the
    transposed V as float values (decode codes with ``e5m2_decode``).  Keys
    are taken in blocks of ``block_n``; the causal mask keeps key j for query
    i iff j <= i.  Returns ``(O [Nq, d], lse [Nq])`` in float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(vt, dtype=np.float64).T
    nq, nk = q.shape[0], k.shape[0]
    c = float(sm_scale) * math.log2(math.e)
    m = np.full(nq, -np.inf)
    l = np.zeros(nq)
    acc = np.zeros((nq, v.shape[1]))
    rows = np.arange(nq)[:, None]
    for j0 in range(0, nk, block_n):
        j1 = min(nk, j0 + block_n)
        qk = q @ k[j0:j1].T
        if causal:
            qk = np.where(np.arange(j0, j1)[None, :] > rows, -np.inf, qk)
        m_new = np.maximum(m, np.max(qk, axis=1) * c)
        live = np.isfinite(m_new)                        # a row that has seen a key
        mb = np.where(live, m_new, 0.0)
        p = np.where(live[:, None], np.exp2(qk * c - mb[:, None]), 0.0)
        alpha = np.where(np.isfinite(m), np.exp2(m - mb), 0.0)
        l = l * alpha + np.sum(p, axis=1)
        acc = acc * alpha[:, None] + e5m2_round(p) @ v[j0:j1]
        m = m_new
    o = acc / l[:, None]
    lse = (m + np.log2(l)) * math.log(2.0)
    return o, lse


def forward_fp8v_heads(q, k, vt, sm_scale: float, causal: bool, heads=None, block_n: int = 128):
    """``forward_fp8v`` over ``[B, H, Nq, d]``, ``[B, H, Nk, d]`` and
    ``[B, H, d, Nk]`` arrays; ``heads`` optionally restricts the work to a
    list of (b, h) pairs (the other outputs are NaN)."""
    q = np.asarray(q, dtype=np.float64)
    B, H, nq, d = q.shape
    o = np.full((B, H, nq, d), np.nan)
    lse = np.full((B, H, nq), np.nan)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    for b, h in heads:
        o[b, h], lse[b, h] = forward_fp8v(q[b, h], k[b, h], vt[b, h], sm_scale, causal, block_n)
    return o, lse
