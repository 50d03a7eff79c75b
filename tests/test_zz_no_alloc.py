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
    # The pointers below are fake device addresses.  Should the size check
    # ever let one through, a launch would follow, so this runs only where no
    # GPU is visible.
    if torch.cuda.is_available():
        pytest.skip("fake device addresses: the size check runs on a machine without a GPU")
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


@pytest.mark.gpu
def test_noalloc_at_the_scratch_limit_allocates_nothing():
    # Exactly FA_NOALLOC_SCRATCH_BYTES of scratch: 16 heads of 131,072 query
    # rows (2,097,152 padded rows), where the entry point's own size check and
    # the backward's workspace check must agree.  Nk is one key tile, so the
    # problem stays small in time.
    rows = fa.NOALLOC_SCRATCH_BYTES // 8
    w = W.custom("bf16", "bhsd", 2, 8, rows // 16, 128, 64, False, seed=73, backward=True)
    assert fa.fa_bwd_workspace_bytes_path(w.B, w.H, w.Nq, w.Nk, w.d,
                                          fa.FA_BWD_PATH_TWO_PASS) == fa.NOALLOC_SCRATCH_BYTES
    x = W.make_inputs(w, device="cuda")
    o, lse = fa.attention_forward(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
    # fa_bwd_noalloc always takes the two-pass backward: the same path through
    # the existing entry point gives bitwise the same gradients
    want = tuple(torch.empty_like(t) for t in (x["q"], x["k"], x["v"]))
    fa.fa_bwd_ex(fa.FA_BWD_PATH_TWO_PASS, 0, x["q"], x["k"], x["v"], o, x["do"], lse, *want, w.sm_scale, w.causal)
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (x["q"], x["k"], x["v"]))
    stream = torch.cuda.current_stream().cuda_stream
    L = fa.lib()

    def call():
        return L.fa_bwd_noalloc(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), o.data_ptr(),
                                x["do"].data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                w.B, w.H, w.Nq, w.Nk, w.d, w.sm_scale, int(w.causal), fa.FA_BF16, stream)

    assert call() == fa.FA_OK   # warm-up: kernels loaded, scratch address looked up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    dq.fill_(float("nan"))
    dk.fill_(float("nan"))
    dv.fill_(float("nan"))
    assert call() == fa.FA_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0, (free0, free1)
    rc, detail = fa.fa_last_device_error()
    assert rc == fa.FA_OK, f"device error {detail:#x}"
    for name, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), want):
        assert torch.equal(a, b), name
    # one query tile more is refused before anything runs
    assert L.fa_bwd_noalloc(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), o.data_ptr(),
                            x["do"].data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                            w.B, w.H, w.Nq + 1, w.Nk, w.d, w.sm_scale, 0, fa.FA_BF16, stream) == fa.FA_ERR_WORKSPACE
