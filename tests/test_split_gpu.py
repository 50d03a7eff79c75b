"""Split-KV forward parity: fa_fwd_split (partial softmaxes over key ranges
merged by their log-sum-exps) against the float64 oracle, element by element,
with the forward's tolerances; edge cases where splits see no keys."""

import pytest
import torch

from tiled_attention_07_gb300 import fa
from tiled_attention_07_gb300 import workloads as W

from parity import check_fwd_head, sample_heads

pytestmark = pytest.mark.gpu


def run_split(w, x, n_splits, guard=4096):
    """fa_fwd_split with NaN-prefilled outputs inside guard regions, and a
    NaN-prefilled workspace (the partial results must be written before use)."""
    q, k, v = x["q"], x["k"], x["v"]
    n = q.numel()
    obuf = torch.full((n + 2 * guard,), float("nan"), dtype=q.dtype, device=q.device)
    o = obuf[guard:guard + n].view(q.shape)
    B, H, Nq, d = fa._dims(q)
    lbuf = torch.full((B * H * Nq + 2 * guard,), float("nan"), dtype=torch.float32, device=q.device)
    lse = lbuf[guard:guard + B * H * Nq].view(B, H, Nq)
    ws = None
    nbytes = fa.fa_fwd_split_workspace_bytes(B, H, Nq, d, n_splits)
    if nbytes:
        ws = torch.full((nbytes // 4,), float("nan"), dtype=torch.float32, device=q.device)
    fa.fa_fwd_split(q, k, v, o, lse, w.sm_scale, w.causal, n_splits, ws)
    torch.cuda.synchronize()
    rc, detail = fa.fa_last_device_error()
    assert rc == fa.FA_OK, f"device error {detail:#x}"
    assert torch.isnan(obuf[:guard]).all() and torch.isnan(obuf[-guard:]).all(), "O guard overwritten"
    assert torch.isnan(lbuf[:guard]).all() and torch.isnan(lbuf[-guard:]).all(), "LSE guard overwritten"
    return o, lse


def check(w, n_splits, heads_limit=10 ** 9):
    x = W.make_inputs(w, device="cuda")
    o, lse = run_split(w, x, n_splits)
    stats = {}
    for b, h in sample_heads(w, heads_limit):
        check_fwd_head(w, x, o, lse, b, h, stats)
    return stats


@pytest.mark.parametrize("name,n_splits", [
    ("fp16_h16_nq1000_nk2500_d80", 4),    # underfilled grid; ragged key tail (Nk = 2500)
    ("fp16_h16_nq1000_nk2500_d80", 20),   # one key tile per split
    ("bf16_b4_h12_n512_d64_causal", 2),   # causal: early query tiles see no key of split 1
    ("fp16_h1_n128_d64", 3),              # more splits than key tiles: empty splits
])
def test_named_workloads_all_heads(name, n_splits):
    print(name, n_splits, check(W.WORKLOADS[name], n_splits))


@pytest.mark.parametrize("dtype,layout,B,H,Nq,Nk,d,causal,n_splits", [
    ("bf16", "bhsd", 1, 3, 300, 1100, 128, False, 5),   # d = 128 (in-place kernel), ragged both ways
    ("bf16", "bhsd", 2, 2, 700, 700, 80, True, 3),      # causal, ragged tiles, d = 80
    ("fp16", "bhsd", 1, 2, 129, 77, 64, True, 2),       # one key tile: split 1 empty for everyone
    ("bf16", "shd", 1, 4, 1000, 2500, 80, True, 6),     # [seq, heads, d], causal with Nq < Nk
    ("fp16", "bhsd", 1, 1, 1, 1000, 64, False, 8),      # a single query row
    ("bf16", "bhsd", 1, 40, 256, 2048, 64, True, 2),    # one-tile blocks two to an SM (160 on 152 SMs)
])
def test_edge_cases(dtype, layout, B, H, Nq, Nk, d, causal, n_splits):
    w = W.custom(dtype, layout, B, H, Nq, Nk, d, causal, seed=Nq + Nk + n_splits)
    print(w.name, n_splits, check(w, n_splits))


def test_one_split_equals_fa_fwd_bitwise():
    w = W.custom("bf16", "bhsd", 1, 4, 600, 900, 80, True, seed=4)
    x = W.make_inputs(w, device="cuda")
    o1 = torch.empty_like(x["q"])
    l1 = torch.empty(fa.lse_shape(x["q"]), dtype=torch.float32, device="cuda")
    fa.fa_fwd(x["q"], x["k"], x["v"], o1, l1, w.sm_scale, w.causal)
    o2, l2 = run_split(w, x, 1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_split_count_stays_in_one_wave():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # 8 query tiles x 16 heads = 128 one-tile CTAs unsplit, 20 key tiles
    s = fa.fa_fwd_split_count(1, 16, 1000, 2500, 80, False)
    assert s == max(1, min(sms // 128, 20 // 4))
    assert 128 * s <= max(sms, 128)
    # 4 heads: 32 one-tile CTAs, a split grid of several per query tile
    s = fa.fa_fwd_split_count(1, 4, 1000, 2500, 80, False)
    assert s == max(1, min(sms // 32, 20 // 4))
    assert 32 * s <= max(sms, 32)
    # few key tiles per query tile: no split
    assert fa.fa_fwd_split_count(4, 12, 512, 512, 64, True) == 1
    # the bench workload fills the GPU unsplit
    assert fa.fa_fwd_split_count(4, 32, 8192, 8192, 80, True) == 1


def test_deterministic():
    w = W.WORKLOADS["fp16_h16_nq1000_nk2500_d80"]
    x = W.make_inputs(w, device="cuda")
    o1, l1 = run_split(w, x, 4)
    o2, l2 = run_split(w, x, 4)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
