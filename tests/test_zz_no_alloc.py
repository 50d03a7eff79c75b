"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (for example plugins inside an inference engine that plans every
buffer in advance) are handed only their inputs and outputs, so this entry
point takes its scratch from a fixed array inside the library instead of a
caller workspace.  These tests check, through the C ABI, that it gives the
same dQ, dK, dV as fa_bwd with a caller workspace, on two calls in a row
(the second sees the scratch the first one left behind), and that problems
larger than the fixed array are refused before anything runs.

The file is named so that pytest collects it last.
"""

import os

import numpy as np
import pytest
import torch

from tiled_attention_07_gb300 import fa
from tiled_attention_07_gb300 import workloads as W

from parity import GRAD_TOL, half_ulp, to64


def test_oversized_problem_is_refused_before_launch():
    if not os.path.exists(fa.LIB_PATH):
        from tiled_attention_07_gb300 import build
        build.build()
    L = fa.lib()
    fake = 1 << 20   # never dereferenced: the size check comes first
    rows = fa.NOALLOC_SCRATCH_BYTES // 8
    # one query tile past the limit
    rc = L.fa_bwd_noalloc(*([fake] * 9), 1, 1, rows + 1, 128, 64, 0.125, 0, fa.FA_BF16, None)
    assert rc == fa.FA_ERR_WORKSPACE
    rc = L.fa_bwd_noalloc(*([fake] * 9), 4, 32, 16384 + 128, 128, 64, 0.125, 1, fa.FA_BF16, None)
    assert rc == fa.FA_ERR_WORKSPACE


def _reference_grads(w, x, o, lse):
    """The existing entry point, with a caller-allocated workspace."""
    return fa.attention_backward(x["q"], x["k"], x["v"], o, x["do"], lse, w.sm_scale, w.causal)


def _noalloc_grads(w, x, o, lse):
    dq = torch.full_like(x["q"], float("nan"))
    dk = torch.full_like(x["k"], float("nan"))
    dv = torch.full_like(x["v"], float("nan"))
    fa.fa_bwd_noalloc(x["q"], x["k"], x["v"], o, x["do"], lse, dq, dk, dv, w.sm_scale, w.causal)
    return dq, dk, dv


@pytest.mark.gpu
def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row():
    cases = [
        # a large first call fills much of the scratch; the smaller second one
        # then runs on top of what the first left behind
        W.custom("bf16", "bhsd", 4, 8, 2000, 2000, 80, True, seed=71, backward=True),
        W.custom("fp16", "bhsd", 2, 3, 333, 517, 64, False, std=0.5, seed=72, backward=True),
    ]
    for w in cases:
        x = W.make_inputs(w, device="cuda")
        o, lse = fa.attention_forward(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
        want = _reference_grads(w, x, o, lse)
        got = _noalloc_grads(w, x, o, lse)
        torch.cuda.synchronize()
        rc, detail = fa.fa_last_device_error()
        assert rc == fa.FA_OK, f"device error {detail:#x}"
        tol = GRAD_TOL[w.dtype]
        for name, a, b in zip(("dq", "dk", "dv"), got, want):
            a64, b64 = to64(a), to64(b)
            assert np.isfinite(a64).all(), name
            scale = max(1.0, float(np.abs(b64).max()))
            excess = (np.abs(a64 - b64) - half_ulp(b64, w.dtype)) / scale
            assert excess.max() <= tol, (w.name, name, float(excess.max()))
