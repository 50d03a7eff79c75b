"""Backward parity: fa_bwd (two-pass recompute backward) through the C ABI
against the float64 oracle's dQ, dK, dV, on the bench workload (sampled
heads) and on ragged / causal / strided edge cases."""

import pytest
import torch

from tiled_attention_07_gb300 import fa
from tiled_attention_07_gb300 import workloads as W

from parity import check_bwd_head, sample_heads

pytestmark = pytest.mark.gpu


def run_fwd_bwd(w, x, guard=0):
    o, lse = fa.attention_forward(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
    grads = {}
    bufs = {}
    for name, src in (("dq", x["q"]), ("dk", x["k"]), ("dv", x["v"])):
        if guard:
            n = src.numel()
            buf = torch.full((n + 2 * guard,), float("nan"), dtype=src.dtype, device=src.device)
            grads[name] = buf[guard:guard + n].view(src.shape)
            bufs[name] = buf
        else:
            grads[name] = torch.full_like(src, float("nan"))
    B, H, Nq, d = fa._dims(x["q"])
    Nk = fa._dims(x["k"])[2]
    need = fa.fa_bwd_workspace_bytes(B, H, Nq, Nk, d)
    ws = torch.full((max(need, 16) // 4,), float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, grads["dq"], grads["dk"], grads["dv"], w.sm_scale,
              w.causal, ws)
    torch.cuda.synchronize()
    rc, detail = fa.fa_last_device_error()
    assert rc == fa.FA_OK, f"device error {detail:#x}"
    for name, buf in bufs.items():
        assert torch.isnan(buf[:guard]).all() and torch.isnan(buf[-guard:]).all(), f"{name} guard overwritten"
    return grads


def check(w, heads_limit=10 ** 9, guard=0):
    x = W.make_inputs(w, device="cuda", with_grad_output=True)
    grads = run_fwd_bwd(w, x, guard)
    stats = {}
    for b, h in sample_heads(w, heads_limit):
        check_bwd_head(w, x, grads, b, h, stats)
    return stats


def test_bench_workload_backward_sampled_heads():
    # 8 seeded heads including (0, 0) and (B-1, H-1)
    stats = check(W.WORKLOADS[W.BENCH_WORKLOAD], heads_limit=8)
    print(stats)


def test_long_causal_d64_backward_sampled_heads():
    stats = check(W.WORKLOADS["bf16_b4_h20_n4096_d64_causal"], heads_limit=8)
    print(stats)


EDGE = [
    ("bf16", "bhsd", 1, 1, 128, 128, 64, False),
    ("bf16", "bhsd", 1, 1, 128, 128, 64, True),
    ("fp16", "bhsd", 2, 3, 129, 77, 64, False),
    ("bf16", "bhsd", 2, 2, 300, 1000, 80, True),
    ("bf16", "bhsd", 1, 2, 1000, 300, 128, True),
    ("fp16", "bhsd", 1, 2, 513, 513, 128, True),
    ("bf16", "bhsd", 3, 1, 256, 255, 80, False),
    ("fp16", "shd", 1, 4, 100, 1000, 64, False),
    ("bf16", "shd", 1, 4, 640, 640, 80, True),
    ("bf16", "bhsd", 4, 12, 512, 512, 64, True),
    ("bf16", "bhsd", 1, 1, 1, 1, 64, True),
]


@pytest.mark.parametrize("case", EDGE, ids=["-".join(map(str, c)) for c in EDGE])
def test_edge_cases(case):
    dt, layout, B, H, Nq, Nk, d, causal = case
    w = W.custom(dt, layout, B, H, Nq, Nk, d, causal, std=0.5 if dt == "fp16" else 1.0, seed=Nq * 3 + Nk,
                 backward=True)
    check(w, heads_limit=6, guard=512)


# Enough heads that the backward kernels run blocks that walk work units
# (the heaviest 128-row tile of a head with its lightest) plus one-tile
# blocks for the rest: two or more rounds of units per SM on a 152-SM part.
PERSIST = [
    # dtype, layout, B, H, Nq, Nk, d, causal
    ("bf16", "bhsd", 2, 160, 512, 512, 80, True),
    ("fp16", "bhsd", 1, 200, 384, 384, 64, True),     # three tiles: the middle one alone in its unit
    ("bf16", "bhsd", 1, 320, 700, 500, 80, False),    # ragged, Nq > Nk
    ("bf16", "bhsd", 1, 256, 500, 900, 64, True),     # causal, Nq < Nk: key tiles past every query
]


@pytest.mark.parametrize("case", PERSIST, ids=["-".join(map(str, c)) for c in PERSIST])
def test_persistent_units(case):
    dt, layout, B, H, Nq, Nk, d, causal = case
    w = W.custom(dt, layout, B, H, Nq, Nk, d, causal, std=0.5 if dt == "fp16" else 1.0, seed=Nq + H + 1,
                 backward=True)
    x = W.make_inputs(w, device="cuda", with_grad_output=True)
    grads = run_fwd_bwd(w, x)
    stats = {}
    heads = [(b, h) for b in range(B) for h in range(H)]
    for b, h in heads[:2] + heads[len(heads) // 2:len(heads) // 2 + 2] + heads[-2:]:
        check_bwd_head(w, x, grads, b, h, stats)
    for n in ("dq", "dk", "dv"):
        assert torch.isfinite(grads[n]).all(), n
    grads2 = run_fwd_bwd(w, x)
    # run to run: bitwise on the two-pass path; the fused path (taken where
    # the workspace size says so) sums dQ's float32 shares in varying order
    two_pass = fa.fa_bwd_workspace_bytes(B, H, Nq, Nk, d) == fa.fa_bwd_workspace_bytes_path(
        B, H, Nq, Nk, d, fa.FA_BWD_PATH_TWO_PASS)
    for n in ("dq", "dk", "dv") if two_pass else ("dk", "dv"):
        assert torch.equal(grads[n], grads2[n]), n
    print(w.name, stats)


def test_deterministic():
    w = W.custom("bf16", "bhsd", 2, 3, 700, 900, 80, True, seed=3, backward=True)
    x = W.make_inputs(w, device="cuda")
    g1 = run_fwd_bwd(w, x)
    g2 = run_fwd_bwd(w, x)
    for n in g1:
        assert torch.equal(g1[n], g2[n]), n


def test_no_queries_gives_zero_dk_dv():
    k = torch.randn(1, 2, 200, 64, device="cuda").to(torch.bfloat16)
    q = torch.zeros(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 2, 0, device="cuda")
    dq = torch.empty_like(q)
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(k, float("nan"))
    fa.fa_bwd(q, k, k, q, q, lse, dq, dk, dv, 0.125, False, torch.empty(16, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert torch.all(dk == 0) and torch.all(dv == 0)
    # Through the C ABI, Nq = 0 reads neither lse nor the workspace: both may be null.
    dk.fill_(float("nan"))
    dv.fill_(float("nan"))
    rc = fa.lib().fa_bwd(q.data_ptr(), k.data_ptr(), k.data_ptr(), q.data_ptr(), q.data_ptr(), None, dq.data_ptr(),
                         dk.data_ptr(), dv.data_ptr(), 1, 2, 0, 200, 64, 0.125, 0, fa.FA_BF16, None, 0,
                         torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.all(dk == 0) and torch.all(dv == 0)


def test_phases_in_order_equal_fa_bwd():
    w = W.custom("bf16", "bhsd", 2, 2, 520, 700, 80, True, seed=13, backward=True)
    x = W.make_inputs(w, device="cuda")
    g1 = run_fwd_bwd(w, x)
    o, lse = fa.attention_forward(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(2, 2, 520, 700, 80), dtype=torch.uint8, device="cuda")
    g2 = {n: torch.full_like(g1[n], float("nan")) for n in g1}
    for phase in (fa.FA_BWD_PREPROCESS, fa.FA_BWD_DKDV, fa.FA_BWD_DQ):
        fa.fa_bwd_phase(phase, x["q"], x["k"], x["v"], o, x["do"], lse, g2["dq"], g2["dk"], g2["dv"], w.sm_scale,
                        w.causal, ws)
    torch.cuda.synchronize()
    for n in g1:
        assert torch.equal(g1[n], g2[n]), n
