"""Forward parity: the CUDA library (through the C ABI) against the float64
oracle, element by element, on seeded inputs shaped like the pages'
workloads, plus edge cases, guard regions and determinism."""

import pytest
import torch

from tiled_attention_07_gb300 import fa
from tiled_attention_07_gb300 import workloads as W

from parity import check_fwd_head, sample_heads

pytestmark = pytest.mark.gpu


def run_fwd(w, x, guard=0):
    """Run fa_fwd with NaN-prefilled outputs; with guard > 0 the outputs are
    views into larger buffers whose edges must stay untouched."""
    q, k, v = x["q"], x["k"], x["v"]
    if guard:
        n = q.numel()
        obuf = torch.full((n + 2 * guard,), float("nan"), dtype=q.dtype, device=q.device)
        o = obuf[guard:guard + n].view(q.shape)
        B, H, Nq, _ = fa._dims(q)
        lbuf = torch.full((B * H * Nq + 2 * guard,), float("nan"), dtype=torch.float32, device=q.device)
        lse = lbuf[guard:guard + B * H * Nq].view(B, H, Nq)
    else:
        o = torch.full_like(q, float("nan"))
        lse = torch.full(fa.lse_shape(q), float("nan"), dtype=torch.float32, device=q.device)
    fa.fa_fwd(q, k, v, o, lse, w.sm_scale, w.causal)
    torch.cuda.synchronize()
    rc, detail = fa.fa_last_device_error()
    assert rc == fa.FA_OK, f"device error {detail:#x}"
    if guard:
        assert torch.isnan(obuf[:guard]).all() and torch.isnan(obuf[-guard:]).all(), "O guard overwritten"
        assert torch.isnan(lbuf[:guard]).all() and torch.isnan(lbuf[-guard:]).all(), "LSE guard overwritten"
    return o, lse


def check(w, heads_limit=10 ** 9, guard=0):
    x = W.make_inputs(w, device="cuda")
    o, lse = run_fwd(w, x, guard)
    stats = {}
    for b, h in sample_heads(w, heads_limit):
        check_fwd_head(w, x, o, lse, b, h, stats)
    return stats


@pytest.mark.parametrize("name", ["fp16_h1_n128_d64", "fp16_h16_nq1000_nk2500_d80", "bf16_b4_h12_n512_d64_causal"])
def test_named_workload_all_heads(name):
    stats = check(W.WORKLOADS[name], guard=4096)
    print(name, stats)


def test_long_causal_d64_all_heads():
    # every one of the 80 heads (the forward runs work-unit blocks here)
    stats = check(W.WORKLOADS["bf16_b4_h20_n4096_d64_causal"])
    print(stats)


def test_bench_workload_forward_sampled_heads():
    # 8 seeded heads including (0, 0) and (B-1, H-1), in the bench's launch configuration
    stats = check(W.WORKLOADS[W.BENCH_WORKLOAD], heads_limit=8)
    print(stats)


EDGE = [
    # dtype, layout, B, H, Nq, Nk, d, causal
    ("bf16", "bhsd", 1, 1, 1, 1, 64, False),
    ("bf16", "bhsd", 1, 1, 1, 1, 64, True),
    ("fp16", "bhsd", 2, 3, 129, 77, 64, False),
    ("bf16", "bhsd", 2, 2, 300, 1000, 80, True),    # causal, Nq < Nk (top-left)
    ("bf16", "bhsd", 1, 2, 1000, 300, 128, True),   # causal, Nq > Nk
    ("fp16", "bhsd", 1, 2, 513, 513, 128, True),
    ("bf16", "bhsd", 3, 1, 256, 255, 80, False),
    ("fp16", "shd", 1, 8, 100, 4096, 64, False),    # the pages' cross-attention shapes
    ("fp16", "shd", 1, 5, 4095, 333, 128, False),
    ("bf16", "shd", 1, 4, 640, 640, 80, True),
    ("fp16", "bhsd", 1, 1, 128, 128, 80, False),
    ("bf16", "bhsd", 1, 1, 256, 128, 64, False),
]


@pytest.mark.parametrize("case", EDGE, ids=["-".join(map(str, c)) for c in EDGE])
def test_edge_cases(case):
    dt, layout, B, H, Nq, Nk, d, causal = case
    w = W.custom(dt, layout, B, H, Nq, Nk, d, causal, std=0.5 if dt == "fp16" else 1.0, seed=Nq * 7 + Nk)
    check(w, guard=1024)


# Shapes with enough heads that the separate-P forward (d <= 96) runs blocks
# that walk several work units (two query-tile pairs of one head each, the
# heaviest with the lightest) plus one-item blocks for the rest: two or more
# rounds of units per SM on a 152-SM part.
PERSIST = [
    # dtype, layout, B, H, Nq, Nk, d, causal
    ("bf16", "bhsd", 2, 160, 512, 512, 80, True),    # one pair per unit side, 320 units
    ("fp16", "bhsd", 1, 200, 768, 768, 64, True),    # three pairs: the middle pair alone in its unit
    ("bf16", "bhsd", 1, 256, 700, 700, 80, False),   # ragged Nq whose last pair still has rows in tile 1
    ("bf16", "bhsd", 1, 320, 1024, 1500, 64, True),  # causal with Nq < Nk
]


@pytest.mark.parametrize("case", PERSIST, ids=["-".join(map(str, c)) for c in PERSIST])
def test_persistent_units(case):
    dt, layout, B, H, Nq, Nk, d, causal = case
    w = W.custom(dt, layout, B, H, Nq, Nk, d, causal, std=0.5 if dt == "fp16" else 1.0, seed=Nq + H)
    x = W.make_inputs(w, device="cuda")
    o, lse = run_fwd(w, x, guard=1024)
    stats = {}
    heads = [(b, h) for b in range(B) for h in range(H)]
    for b, h in heads[:2] + heads[len(heads) // 2:len(heads) // 2 + 2] + heads[-2:]:
        check_fwd_head(w, x, o, lse, b, h, stats)
    # every head was written (NaN-free) and equals a second, identical run
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    o2, lse2 = run_fwd(w, x)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    print(w.name, stats)


# d = 64 shapes whose two-tile grid is under one wave while their one-tile
# grid (query tiles x heads) is between one and two blocks per SM on a 152-SM
# part: the forward runs its one-tile build, two blocks to an SM.
TWO_PER_SM = [
    # dtype, layout, B, H, Nq, Nk, d, causal
    ("fp16", "bhsd", 1, 100, 256, 256, 64, False),   # 200 one-tile blocks
    ("bf16", "bhsd", 1, 90, 200, 700, 64, True),     # ragged second tile, causal with Nq < Nk
    ("bf16", "shd", 1, 60, 300, 300, 64, True),      # [seq, heads, d], three tiles per head
    ("fp16", "bhsd", 1, 48, 513, 129, 64, True),     # causal with Nq > Nk: late tiles see every key
]


@pytest.mark.parametrize("case", TWO_PER_SM, ids=["-".join(map(str, c)) for c in TWO_PER_SM])
def test_one_tile_build_two_per_sm(case):
    dt, layout, B, H, Nq, Nk, d, causal = case
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles, pairs = (Nq + 127) // 128, (Nq + 255) // 256
    print("one-tile build taken:", pairs * B * H < sms < tiles * B * H <= 2 * sms)
    w = W.custom(dt, layout, B, H, Nq, Nk, d, causal, std=0.5 if dt == "fp16" else 1.0, seed=Nq + 3 * H)
    x = W.make_inputs(w, device="cuda")
    o, lse = run_fwd(w, x, guard=1024)
    stats = {}
    heads = [(b, h) for b in range(B) for h in range(H)]
    for b, h in heads[:2] + heads[len(heads) // 2:len(heads) // 2 + 1] + heads[-2:]:
        check_fwd_head(w, x, o, lse, b, h, stats)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    o2, lse2 = run_fwd(w, x)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    print(w.name, stats)


def test_large_logits_trigger_rescaling():
    # q, k spread widely so that running maxima jump by more than 2^8 between
    # key tiles (checks the lazy O rescaling); v stays N(0, 1) so that |O|
    # stays in the range the absolute tolerance is stated for
    for w in (W.custom("bf16", "bhsd", 1, 2, 512, 2048, 64, False, sm_scale=1.0, std=2.5, seed=5),
              W.custom("fp16", "bhsd", 1, 2, 384, 1500, 128, True, sm_scale=0.6, std=2.0, seed=6)):
        x = W.make_inputs(w, device="cuda")
        g = torch.Generator().manual_seed(w.seed + 1000)
        x["v"] = torch.randn(x["v"].shape, generator=g).to(x["v"].dtype).cuda()
        o, lse = run_fwd(w, x)
        stats = {}
        for b, h in sample_heads(w, 100):
            check_fwd_head(w, x, o, lse, b, h, stats)


def test_constant_v_gives_constant_o():
    w = W.custom("bf16", "bhsd", 1, 2, 300, 700, 80, True, seed=9)
    x = W.make_inputs(w, device="cuda")
    x["v"] = torch.full_like(x["v"], 1.5)
    o, _ = run_fwd(w, x)
    assert torch.all(o == 1.5)


def test_deterministic():
    w = W.custom("bf16", "bhsd", 2, 3, 700, 900, 80, True, seed=3)
    x = W.make_inputs(w, device="cuda")
    o1, l1 = run_fwd(w, x)
    o2, l2 = run_fwd(w, x)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_empty_query_is_noop():
    q = torch.zeros(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.randn(1, 2, 5, 64, device="cuda").to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 0, device="cuda")
    fa.fa_fwd(q, k, k, o, lse, 0.125, True)
    torch.cuda.synchronize()
