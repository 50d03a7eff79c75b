"""Float64 CPU oracle for the row-wise softmax ("Long Softmax").

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the tests and ``bench.py``'s CPU legs call it.  It shares no code with
the CUDA library.

"Puzzles 8 Long Softmax": z_ij = softmax(x_i1, ..., x_iT)_j for every row i,
made numerically stable by subtracting the row max.  The puzzle's online
version (max and sum loops merged by rescaling the running sum) reaches the
same value up to rounding, so the oracle is the plain definition in float64:

    m_i = max_j x_ij,  s_i = sum_j exp(x_ij - m_i),
    z_ij = exp(x_ij - m_i) / s_i,  lse_i = m_i + log s_i.

Reading taken where the pages are open: every element of a row takes part in
the sum (the puzzle's listing pads the last tile with zeros, which would add
exp(0 - m) per padded slot; the definition has no padding).

Parity: pinned (see tests/test_oracle_softmax.py): brute force at 50 digits,
closed forms, invariants.
"""

from __future__ import annotations

import numpy as np

__all__ = ["softmax_rows"]


def softmax_rows(x):
    """Row softmax and row log-sum-exp of a [rows, T] matrix, in float64.

    Returns ``(z [rows, T], lse [rows])``.  Entries of -inf get z = 0; a row
    of -inf only is undefined (NaN), as the definition is.
    """
    x = np.asarray(x, dtype=np.float64)
    if x.ndim != 2:
        raise ValueError("expected a [rows, T] matrix")
    with np.errstate(invalid="ignore"):
        m = np.max(x, axis=1)
        e = np.exp(x - m[:, None])
        s = np.sum(e, axis=1)
        z = e / s[:, None]
        lse = m + np.log(s)
    return z, lse
