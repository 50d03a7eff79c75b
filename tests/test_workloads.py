"""Host-side checks of the seeded input generators and the work accounting."""

import math

import torch

from tiled_attention_07_gb300 import workloads as W


def test_named_workloads_match_their_shapes():
    c1 = W.WORKLOADS["fp16_h1_n128_d64"]
    x = W.make_inputs(c1)
    assert x["q"].shape == (128, 1, 64) and x["q"].dtype == torch.float16
    c2 = W.WORKLOADS["fp16_h16_nq1000_nk2500_d80"]
    assert c2.shape(c2.Nq) == (1000, 16, 80) and c2.shape(c2.Nk) == (2500, 16, 80)
    c5 = W.WORKLOADS[W.BENCH_WORKLOAD]
    assert c5.backward and c5.causal and c5.shape(c5.Nq) == (4, 32, 8192, 80)
    assert abs(c5.sm_scale - 1 / math.sqrt(80)) < 1e-15


def test_generator_is_seeded_and_distribution_is_right():
    w = W.custom("bf16", "bhsd", 2, 3, 300, 200, 64, False, std=0.5, seed=7, backward=True)
    a = W.make_inputs(w)
    b = W.make_inputs(w)
    for key in ("q", "k", "v", "do"):
        assert torch.equal(a[key], b[key])
    q = a["q"].float()
    assert abs(q.std().item() - 0.5) < 0.01 and abs(q.mean().item()) < 0.01
    assert abs(a["do"].float().std().item() - 1.0) < 0.02
    assert not torch.equal(a["q"], a["k"])


def test_flop_accounting():
    w = W.custom("bf16", "bhsd", 4, 32, 8192, 8192, 80, True)
    assert w.fwd_flops() == 4 * 4 * 32 * 8192 * 8192 * 80 / 2
    assert w.bwd_flops() == 2.5 * w.fwd_flops()
    w2 = W.custom("fp16", "shd", 1, 16, 1000, 2500, 80, False)
    assert w2.fwd_flops() == 4 * 16 * 1000 * 2500 * 80


def test_fp8v_inputs_layout_and_padding():
    import numpy as np

    import oracle.fp8 as ref8

    w = W.custom("fp16", "bhsd", 2, 3, 40, 70, 64, True, seed=5)
    x = W.fp8v_inputs(w, ld=96, pad_code=0x7F)
    vt, v8 = x["vt"], x["v8"]
    assert vt.dtype == torch.uint8 and vt.shape == (2, 3, 64, 96)
    assert v8.shape == (2, 3, 70, 64) and v8.dtype == torch.float32
    assert torch.all(vt[..., 70:] == 0x7F)                       # bytes past Nk hold the pad code
    # vt[b, h, c, j] is the e5m2 code of v8[b, h, j, c]
    dec = ref8.e5m2_decode(vt[..., :70].numpy())
    assert np.array_equal(dec, v8.transpose(-1, -2).numpy().astype(np.float64))
    # the codes are V of make_inputs rounded to e5m2: within the format's 2^-3 relative step
    v = W.make_inputs(w)["v"].float()
    assert torch.all((v8 - v).abs() <= 2.0 ** -3 * v.abs() + 2.0 ** -17)
    # default row length: Nk rounded up to 16
    assert W.fp8v_inputs(w)["vt"].shape[-1] == 80


def test_algorithmic_bytes_match_the_configuration_table():
    # fwd: q, k, v read and o written once (2 bytes each) plus the fp32 LSE;
    # bwd: q, k, v, o, dO read and dq, dk, dv written, plus LSE and D per row
    mb = {n: W.WORKLOADS[n].fwd_bytes() / 1e6 for n in W.WORKLOADS}
    assert abs(mb["fp16_h16_nq1000_nk2500_d80"] - 17.98) < 0.01
    assert abs(mb["bf16_b4_h12_n512_d64_causal"] - 12.68) < 0.01
    assert abs(mb["bf16_b4_h20_n4096_d64_causal"] - 169.08) < 0.01
    assert abs(mb[W.BENCH_WORKLOAD] - 675.28) < 0.01
    assert abs(W.WORKLOADS[W.BENCH_WORKLOAD].bwd_bytes() / 1e9 - 1.3506) < 1e-4
    # the causal mask halves the work, not the bytes
    w = W.custom("bf16", "bhsd", 1, 1, 256, 256, 64, True)
    assert w.fwd_bytes() == W.custom("bf16", "bhsd", 1, 1, 256, 256, 64, False).fwd_bytes()
