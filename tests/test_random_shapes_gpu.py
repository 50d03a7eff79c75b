"""Seeded random shapes through the forward and backward, against the float64
oracle: dtype, layout, head dim, causal mask, ragged Nq and Nk, and head
counts up to a few hundred (enough for the forward's work-unit blocks) drawn
from a fixed seed, so every run checks the same cases."""

import random

import pytest
import torch

from tiled_attention_07_gb300 import fa
from tiled_attention_07_gb300 import workloads as W

from parity import check_bwd_head, check_fwd_head

pytestmark = pytest.mark.gpu


def cases(n, seed=2026):
    rnd = random.Random(seed)
    out = []
    for i in range(n):
        dtype = rnd.choice(["fp16", "bf16"])
        d = rnd.choice([64, 80, 128])
        layout = rnd.choice(["bhsd", "bhsd", "shd"])
        causal = rnd.random() < 0.6
        nq = rnd.choice([rnd.randint(1, 300), rnd.randint(300, 1500)])
        nk = nq if (causal and rnd.random() < 0.5) else rnd.choice([rnd.randint(1, 300), rnd.randint(300, 1500)])
        if layout == "shd":
            b, h = 1, rnd.choice([1, 3, 8])
        elif rnd.random() < 0.3:
            b, h = rnd.choice([1, 2]), rnd.choice([160, 200, 320])   # many heads
            nq = nk = rnd.choice([256, 384, 512, 700])
        else:
            b, h = rnd.randint(1, 3), rnd.randint(1, 5)
        out.append((i, dtype, layout, b, h, nq, nk, d, causal))
    return out


CASES = cases(16)


@pytest.mark.parametrize("case", CASES, ids=["-".join(map(str, c)) for c in CASES])
def test_random_shape_forward_backward(case):
    i, dtype, layout, B, H, Nq, Nk, d, causal = case
    w = W.custom(dtype, layout, B, H, Nq, Nk, d, causal, std=0.5 if dtype == "fp16" else 1.0, seed=100 + i,
                 backward=True)
    x = W.make_inputs(w, device="cuda", with_grad_output=True)
    o, lse = fa.attention_forward(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
    dq, dk, dv = fa.attention_backward(x["q"], x["k"], x["v"], o, x["do"], lse, w.sm_scale, w.causal)
    torch.cuda.synchronize()
    rc, detail = fa.fa_last_device_error()
    assert rc == fa.FA_OK, f"device error {detail:#x}"
    heads = [(b, h) for b in range(B) for h in range(H)]
    pick = heads if len(heads) <= 3 else [heads[0], heads[len(heads) // 2], heads[-1]]
    stats = {}
    for b, h in pick:
        check_fwd_head(w, x, o, lse, b, h, stats)
        check_bwd_head(w, x, {"dq": dq, "dk": dk, "dv": dv}, b, h, stats)
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t).all()
    print(w.name, stats)
