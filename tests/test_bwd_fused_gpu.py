"""The fused backward (FA_BWD_PATH_FUSED, d = 64) through the C ABI.

One pass over key tiles forms dK, dV and each query tile's share of dQ
("[CS336] Assignment 2: Systems", "FlashAttention V2 / Backward Pass": dQ
accumulates along key tiles, dK and dV along query tiles; here the dQ shares
are summed in a float32 accumulator instead of a second pass).  Checked
against the float64 oracle with the backward bounds of tests/parity.py, and
against the two-pass path: dK and dV come from the same arithmetic and must
be bitwise equal; dQ is summed in another order and is compared by the
oracle bounds only.
"""

import pytest
import torch

from tiled_attention_07_gb300 import fa
from tiled_attention_07_gb300 import workloads as W

from parity import check_bwd_head, sample_heads

pytestmark = pytest.mark.gpu


def _grads(w, x, o, lse, path, guard=0, phases=False):
    out, bufs = {}, {}
    for name, src in (("dq", x["q"]), ("dk", x["k"]), ("dv", x["v"])):
        if guard:
            n = src.numel()
            buf = torch.full((n + 2 * guard,), float("nan"), dtype=src.dtype, device=src.device)
            out[name] = buf[guard:guard + n].view(src.shape)
            bufs[name] = buf
        else:
            out[name] = torch.full_like(src, float("nan"))
    B, H, Nq, d = fa._dims(x["q"])
    Nk = fa._dims(x["k"])[2]
    need = fa.fa_bwd_workspace_bytes_path(B, H, Nq, Nk, d, path)
    ws = torch.full((max(need, 16) // 4,), float("nan"), dtype=torch.float32, device="cuda")
    args = (x["q"], x["k"], x["v"], o, x["do"], lse, out["dq"], out["dk"], out["dv"], w.sm_scale, w.causal, ws)
    if phases:
        for ph in (fa.FA_BWD_PREPROCESS, fa.FA_BWD_DKDV, fa.FA_BWD_DQ):
            fa.fa_bwd_ex(path, ph, *args)
    else:
        fa.fa_bwd_ex(path, 0, *args)
    torch.cuda.synchronize()
    rc, detail = fa.fa_last_device_error()
    assert rc == fa.FA_OK, f"device error {detail:#x}"
    for name, buf in bufs.items():
        assert torch.isnan(buf[:guard]).all() and torch.isnan(buf[-guard:]).all(), f"{name} guard overwritten"
    return out


def _check(w, heads_limit=8, guard=0):
    x = W.make_inputs(w, device="cuda", with_grad_output=True)
    o, lse = fa.attention_forward(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
    fused = _grads(w, x, o, lse, fa.FA_BWD_PATH_FUSED, guard=guard)
    two = _grads(w, x, o, lse, fa.FA_BWD_PATH_TWO_PASS)
    for n in ("dk", "dv"):
        assert torch.equal(fused[n], two[n]), f"{n} differs from the two-pass path"
    stats = {}
    for b, h in sample_heads(w, heads_limit):
        check_bwd_head(w, x, fused, b, h, stats)
    return stats


def test_long_causal_d64_backward_sampled_heads():
    # the d = 64 long causal shape (B4 H20 N4096), 8 seeded heads
    print(_check(W.WORKLOADS["bf16_b4_h20_n4096_d64_causal"], heads_limit=8))


EDGE = [
    # dtype, layout, B, H, Nq, Nk, causal
    ("bf16", "bhsd", 1, 1, 128, 128, False),
    ("bf16", "bhsd", 1, 1, 128, 128, True),
    ("fp16", "bhsd", 2, 3, 129, 77, False),      # ragged, one key tile with a tail
    ("bf16", "bhsd", 2, 2, 300, 1000, True),     # Nq < Nk: key tiles past every query
    ("bf16", "bhsd", 1, 2, 1000, 300, True),     # Nq > Nk
    ("fp16", "bhsd", 1, 2, 513, 513, True),
    ("bf16", "bhsd", 3, 1, 256, 255, False),
    ("fp16", "shd", 1, 4, 100, 1000, False),     # [seq, heads, d]
    ("bf16", "shd", 1, 4, 640, 640, True),
    ("bf16", "bhsd", 4, 12, 512, 512, True),     # the short causal d = 64 shape
    ("bf16", "bhsd", 1, 1, 1, 1, True),
    ("bf16", "bhsd", 1, 160, 700, 700, True),    # many heads
]


@pytest.mark.parametrize("case", EDGE, ids=["-".join(map(str, c)) for c in EDGE])
def test_edge_cases(case):
    dt, layout, B, H, Nq, Nk, causal = case
    w = W.custom(dt, layout, B, H, Nq, Nk, 64, causal, std=0.5 if dt == "fp16" else 1.0, seed=Nq * 7 + Nk,
                 backward=True)
    _check(w, heads_limit=4, guard=512)


def test_phases_in_order_equal_the_whole_call():
    w = W.custom("bf16", "bhsd", 2, 2, 520, 700, 64, True, seed=17, backward=True)
    x = W.make_inputs(w, device="cuda")
    o, lse = fa.attention_forward(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
    g1 = _grads(w, x, o, lse, fa.FA_BWD_PATH_FUSED)
    g2 = _grads(w, x, o, lse, fa.FA_BWD_PATH_FUSED, phases=True)
    for n in ("dk", "dv"):
        assert torch.equal(g1[n], g2[n]), n
    stats = {}
    for b, h in sample_heads(w, 4):
        check_bwd_head(w, x, g2, b, h, stats)


def test_repeat_runs_agree():
    # dK, dV bitwise; dQ within the oracle bounds on both runs (its float32
    # additions may come in another order)
    w = W.custom("bf16", "bhsd", 2, 3, 700, 900, 64, True, seed=3, backward=True)
    x = W.make_inputs(w, device="cuda")
    o, lse = fa.attention_forward(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
    g1 = _grads(w, x, o, lse, fa.FA_BWD_PATH_FUSED)
    g2 = _grads(w, x, o, lse, fa.FA_BWD_PATH_FUSED)
    for n in ("dk", "dv"):
        assert torch.equal(g1[n], g2[n]), n
    for g in (g1, g2):
        stats = {}
        for b, h in sample_heads(w, 3):
            check_bwd_head(w, x, g, b, h, stats)


def test_errors_and_auto_selection():
    w = W.custom("bf16", "bhsd", 1, 2, 256, 256, 80, True, seed=5, backward=True)
    x = W.make_inputs(w, device="cuda")
    o, lse = fa.attention_forward(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
    dq, dk, dv = (torch.empty_like(t) for t in (x["q"], x["k"], x["v"]))
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:   # no fused path at d = 80
        fa.fa_bwd_ex(fa.FA_BWD_PATH_FUSED, 0, x["q"], x["k"], x["v"], o, x["do"], lse, dq, dk, dv, w.sm_scale,
                     w.causal, ws)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_bwd_workspace_bytes_path(1, 2, 256, 256, 80, fa.FA_BWD_PATH_FUSED) == 0
    # d = 64: a two-pass-sized workspace is too small for the fused path, and
    # under AUTO it selects the two-pass path
    w = W.custom("bf16", "bhsd", 1, 2, 256, 256, 64, True, seed=5, backward=True)
    x = W.make_inputs(w, device="cuda")
    o, lse = fa.attention_forward(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
    small = fa.fa_bwd_workspace_bytes_path(1, 2, 256, 256, 64, fa.FA_BWD_PATH_TWO_PASS)
    assert fa.fa_bwd_workspace_bytes_path(1, 2, 256, 256, 64, fa.FA_BWD_PATH_FUSED) == small // 8 * 4 * (2 + 64)
    ws = torch.empty(small, dtype=torch.uint8, device="cuda")
    out = {n: torch.empty_like(x[s]) for n, s in (("dq", "q"), ("dk", "k"), ("dv", "v"))}
    with pytest.raises(fa.FaError) as e:
        fa.fa_bwd_ex(fa.FA_BWD_PATH_FUSED, 0, x["q"], x["k"], x["v"], o, x["do"], lse, out["dq"], out["dk"],
                     out["dv"], w.sm_scale, w.causal, ws)
    assert e.value.code == fa.FA_ERR_WORKSPACE
    fa.fa_bwd_ex(fa.FA_BWD_PATH_AUTO, 0, x["q"], x["k"], x["v"], o, x["do"], lse, out["dq"], out["dk"], out["dv"],
                 w.sm_scale, w.causal, ws)
    two = _grads(w, x, o, lse, fa.FA_BWD_PATH_TWO_PASS)
    torch.cuda.synchronize()
    for n in ("dq", "dk", "dv"):
        assert torch.equal(out[n], two[n]), n
