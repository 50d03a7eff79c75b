"""Forward with V in float8 e5m2 (fa_fwd_fp8v) against the float64 oracles.

Two comparisons:

* Tight, against the e5m2 oracle (oracle.fp8.forward_fp8v), with the
  forward's tolerances.  The inputs put every row's largest score at key 0
  (q = (1, r_i), k_0 = (a, 0, ...), k_j = (0, t_j)), so the running max is
  final after the first key tile, on the GPU (which keeps its max unless it
  grows) as in the oracle (which updates it every tile): both cast the same p
  to e5m2.  Rows where a random score comes within 1e-3 of key 0's are left
  out of this check (at least 90 % must remain).  The GPU result must also be
  nearer the e5m2 oracle than the exact one, so the cast is really there.
* Loose, against the exact oracle on plain random inputs: the cast of p
  (relative error <= 2^-3) bounds |O_gpu - O_exact| by 2^-3 max |v| over the
  row's visible keys, plus the 16-bit tolerance and half an output ulp; the
  LSE sums unrounded p and keeps the forward's LSE tolerance.
"""

import numpy as np
import pytest
import torch

import oracle.attention as ref
import oracle.fp8 as ref8
from tiled_attention_07_gb300 import fa
from tiled_attention_07_gb300 import workloads as W

from parity import LSE_TOL, O_TOL, half_ulp, to64

pytestmark = pytest.mark.gpu


def run(w, x):
    q, k, vt = x["q"], x["k"], x["vt"]
    o = torch.full_like(q, float("nan"))
    lse = torch.full(fa.lse_shape(q), float("nan"), dtype=torch.float32, device=q.device)
    fa.fa_fwd_fp8v(q, k, vt, o, lse, w.sm_scale, w.causal)
    torch.cuda.synchronize()
    rc, detail = fa.fa_last_device_error()
    assert rc == fa.FA_OK, f"device error {detail:#x}"
    return o, lse


def key0_max_inputs(w, device="cuda", pad_code=0):
    """fp8v_inputs with every row's largest score at key 0 (see above)."""
    x = W.fp8v_inputs(w, "cpu", pad_code=pad_code)
    q, k = x["q"].clone(), x["k"].clone()
    a = 5.0 / w.sm_scale
    q[..., 0] = 1.0
    k[..., 0] = 0.0
    k[..., 0, :] = 0.0
    k[..., 0, 0] = a
    x["q"], x["k"] = q, k
    return {n: t.to(device) for n, t in x.items()}


def oracle_heads(w, x, heads, exact=False):
    out = {}
    for b, h in heads:
        q = to64(x["q"][b, h])
        k = to64(x["k"][b, h])
        vt = to64(x["v8"][b, h]).T
        if exact:
            out[(b, h)] = ref.forward(q, k, vt.T, w.sm_scale, w.causal)
        else:
            out[(b, h)] = ref8.forward_fp8v(q, k, vt, w.sm_scale, w.causal)
    return out


def heads_of(w, limit=4):
    hs = [(b, h) for b in range(w.B) for h in range(w.H)]
    return hs if len(hs) <= limit else [hs[0], hs[len(hs) // 2], hs[-1]]


def check_tight(w):
    x = key0_max_inputs(w)
    o, lse = run(w, x)
    heads = heads_of(w)
    r8 = oracle_heads(w, x, heads)
    rx = oracle_heads(w, x, heads, exact=True)
    kept = total = 0
    d8 = dx = 0.0
    for b, h in heads:
        o8, l8 = r8[(b, h)]
        ox, lx = rx[(b, h)]
        og = to64(o[b, h])
        # rows whose maximum is key 0 by a margin
        s = ref.scores(to64(x["q"][b, h]), to64(x["k"][b, h]), w.sm_scale, w.causal)
        others = np.max(np.where(np.arange(s.shape[1])[None, :] == 0, -np.inf, s), axis=1)
        rows = s[:, 0] > others + 1e-3
        kept += int(rows.sum())
        total += rows.size
        err = np.abs(og - o8)[rows] - half_ulp(o8[rows], w.dtype)
        assert err.max() <= O_TOL[w.dtype], f"head {(b, h)}: max |O - O_e5m2| excess {err.max():.3g}"
        assert np.abs(to64(lse[b, h]) - lx).max() <= LSE_TOL
        d8 += float(np.sum((og - o8)[rows] ** 2))
        dx += float(np.sum((og - ox)[rows] ** 2))
    assert kept >= 0.9 * total, f"only {kept} of {total} rows have their maximum at key 0"
    assert d8 < 0.25 * dx, f"GPU not nearer the e5m2 oracle than the exact one ({d8:.3g} vs {dx:.3g})"
    return {"rows": kept, "rms_vs_e5m2": (d8 / kept / w.d) ** 0.5, "rms_vs_exact": (dx / kept / w.d) ** 0.5}


def check_loose(w, pad_code=0):
    x = W.fp8v_inputs(w, "cuda", pad_code=pad_code)
    o, lse = run(w, x)
    heads = heads_of(w)
    rx = oracle_heads(w, x, heads, exact=True)
    worst = 0.0
    for b, h in heads:
        ox, lx = rx[(b, h)]
        og = to64(o[b, h])
        v = to64(x["v8"][b, h])                       # [Nk, d]
        absmax = np.maximum.accumulate(np.max(np.abs(v), axis=1))   # max |v| over keys 0..j
        vis = np.minimum(np.arange(w.Nq), w.Nk - 1) if w.causal else np.full(w.Nq, w.Nk - 1)
        bound = 2.0 ** -3 * absmax[vis][:, None] + O_TOL[w.dtype] + half_ulp(ox, w.dtype)
        assert np.all(np.abs(og - ox) <= bound), f"head {(b, h)}: beyond the e5m2 cast bound"
        assert np.abs(to64(lse[b, h]) - lx).max() <= LSE_TOL
        worst = max(worst, float(np.max(np.abs(og - ox) / bound)))
    return {"worst_fraction_of_bound": worst}


@pytest.mark.parametrize("dtype,B,H,Nq,Nk,d,causal", [
    ("fp16", 1, 2, 500, 1000, 64, False),
    ("fp16", 1, 2, 700, 700, 80, True),
    ("fp16", 2, 1, 300, 300, 80, False),     # ragged key tail, ld = 304
    ("bf16", 1, 3, 640, 640, 64, True),
    ("fp16", 1, 2, 513, 700, 128, False),    # d = 128: P over the S columns
    ("fp16", 2, 1, 600, 600, 128, True),
    ("fp16", 1, 320, 512, 512, 80, True),    # enough heads for the work-unit blocks
])
def test_tight_against_e5m2_oracle(dtype, B, H, Nq, Nk, d, causal):
    w = W.custom(dtype, "bhsd", B, H, Nq, Nk, d, causal, seed=Nq + Nk + d)
    print(w.name, check_tight(w))


@pytest.mark.parametrize("dtype,B,H,Nq,Nk,d,causal", [
    ("bf16", 1, 2, 1024, 1024, 80, True),
    ("fp16", 1, 2, 1000, 2500, 80, False),   # the cross-attention shape, ragged keys
    ("bf16", 2, 2, 129, 77, 64, True),       # one ragged key tile
    ("fp16", 1, 1, 1, 1000, 64, False),      # a single query row
    ("bf16", 1, 2, 1000, 1000, 128, True),
    ("bf16", 2, 160, 768, 768, 64, True),    # work-unit blocks, an odd middle pair
])
def test_loose_against_exact(dtype, B, H, Nq, Nk, d, causal):
    w = W.custom(dtype, "bhsd", B, H, Nq, Nk, d, causal, seed=3 * Nq + Nk)
    print(w.name, check_loose(w))


def test_padding_bytes_are_not_read():
    # Row bytes past Nk hold e5m2 NaN codes: any read of them would reach O.
    w = W.custom("fp16", "bhsd", 1, 2, 256, 200, 64, False, seed=9)
    x = W.fp8v_inputs(w, "cuda", ld=256, pad_code=0x7F)
    o, lse = run(w, x)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    print(check_loose(w, pad_code=0x7F))
