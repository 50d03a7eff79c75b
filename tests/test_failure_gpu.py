"""Failure detection without a GPU fault: the device error word set from the
host makes every bounded wait of the real kernels give up at once; the kernels
must still finish, the status must come back as FA_ERR_TIMEOUT, and the next
calls on the same context must be correct again."""

import pytest
import torch

from tiled_attention_07_gb300 import fa
from tiled_attention_07_gb300 import workloads as W

from parity import check_bwd_head, check_fwd_head

pytestmark = pytest.mark.gpu


def test_injected_give_up_is_reported_and_context_stays_usable():
    w = W.custom("bf16", "bhsd", 1, 2, 700, 900, 80, True, seed=31, backward=True)
    x = W.make_inputs(w, device="cuda")
    assert fa.fa_last_device_error() == (fa.FA_OK, 0)
    # forward with the word set: finishes, reports the injected code
    fa.fa_inject_device_error(0x1234)
    o, lse = fa.attention_forward(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
    rc, detail = fa.fa_last_device_error()
    assert rc == fa.FA_ERR_TIMEOUT and detail == 0x1234
    # the word was cleared: the same call is correct now
    o, lse = fa.attention_forward(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
    assert fa.fa_last_device_error() == (fa.FA_OK, 0)
    stats = {}
    for h in range(w.H):
        check_fwd_head(w, x, o, lse, 0, h, stats)
    # backward (three launches) with the word set
    fa.fa_inject_device_error(0x77)
    fa.attention_backward(x["q"], x["k"], x["v"], o, x["do"], lse, w.sm_scale, w.causal)
    rc, detail = fa.fa_last_device_error()
    assert rc == fa.FA_ERR_TIMEOUT and detail == 0x77
    grads = dict(zip(("dq", "dk", "dv"), fa.attention_backward(x["q"], x["k"], x["v"], o, x["do"], lse,
                                                              w.sm_scale, w.causal)))
    assert fa.fa_last_device_error() == (fa.FA_OK, 0)
    for h in range(w.H):
        check_bwd_head(w, x, grads, 0, h, stats)
    torch.cuda.synchronize()
