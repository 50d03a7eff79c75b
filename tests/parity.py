"""Helpers for the CUDA-vs-oracle parity tests.

Tolerances (stated for the forward by the workload definition, derived for
the backward):

* forward O: max |O_gpu - O_ref| <= 2e-3 (fp16) / 1e-2 (bf16), where each
  element may in addition be off by half an ulp of the output type at
  |O_ref| (the rounding of a correct result to fp16/bf16 alone reaches
  0.0156 for bf16 values in [4, 8)); the plain max is reported as well.
* forward LSE: max |LSE_gpu - LSE_ref| <= 1e-3.
* backward dQ, dK, dV: max |d_gpu - d_ref| <= tol * max(1, max |d_ref|) with
  tol = 2e-3 (fp16) / 1e-2 (bf16), plus half an output ulp per element.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle.attention as ref
from tiled_attention_07_gb300 import workloads as W

O_TOL = {"fp16": 2e-3, "bf16": 1e-2}
LSE_TOL = 1e-3
GRAD_TOL = {"fp16": 2e-3, "bf16": 1e-2}
MANTISSA_BITS = {"fp16": 10, "bf16": 7}


def half_ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Half an ulp of the 16-bit type at |x| (x in float64)."""
    ax = np.abs(x)
    _, e = np.frexp(np.where(ax > 0, ax, 1.0))
    ulp = np.ldexp(1.0, e - 1 - MANTISSA_BITS[dtype])
    return np.where(ax > 0, 0.5 * ulp, 0.0)


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def head(t: torch.Tensor, w: W.Workload, b: int, h: int) -> np.ndarray:
    return to64(W.head_view(t, w.layout, b, h))


def sample_heads(w: W.Workload, limit: int):
    """All (b, h) pairs, or a seeded sample of `limit` of them that always
    includes the first and the last."""
    allp = [(b, h) for b in range(w.B) for h in range(w.H)]
    if len(allp) <= limit:
        return allp
    rng = np.random.default_rng(w.seed)
    mid = [allp[i] for i in sorted(rng.choice(np.arange(1, len(allp) - 1), size=limit - 2, replace=False))]
    return [allp[0]] + mid + [allp[-1]]


def check_fwd_head(w: W.Workload, x: dict, o: torch.Tensor, lse: torch.Tensor, b: int, h: int, stats: dict):
    q, k, v = head(x["q"], w, b, h), head(x["k"], w, b, h), head(x["v"], w, b, h)
    o_ref, lse_ref = ref.forward(q, k, v, w.sm_scale, w.causal)
    o_gpu = head(o, w, b, h)
    lse_gpu = to64(lse[b, h])
    assert np.isfinite(o_gpu).all(), f"non-finite O at head {(b, h)}"
    assert np.isfinite(lse_gpu).all(), f"non-finite LSE at head {(b, h)}"
    err = np.abs(o_gpu - o_ref)
    excess = err - half_ulp(o_ref, w.dtype)
    stats["max_dO"] = max(stats.get("max_dO", 0.0), float(err.max()))
    stats["max_dO_minus_half_ulp"] = max(stats.get("max_dO_minus_half_ulp", -1.0), float(excess.max()))
    stats["max_dLSE"] = max(stats.get("max_dLSE", 0.0), float(np.abs(lse_gpu - lse_ref).max()))
    tol = O_TOL[w.dtype]
    if excess.max() > tol:
        i = np.unravel_index(np.argmax(excess), excess.shape)
        raise AssertionError(f"O mismatch at head {(b, h)} row {i[0]} col {i[1]}: gpu {o_gpu[i]} ref {o_ref[i]} "
                             f"(|d| = {err[i]:.3g} > {tol} + half ulp)")
    dl = np.abs(lse_gpu - lse_ref)
    if dl.max() > LSE_TOL:
        i = int(np.argmax(dl))
        raise AssertionError(f"LSE mismatch at head {(b, h)} row {i}: gpu {lse_gpu[i]} ref {lse_ref[i]}")


def check_bwd_head(w: W.Workload, x: dict, grads: dict, b: int, h: int, stats: dict):
    q, k, v, do = (head(x[n], w, b, h) for n in ("q", "k", "v", "do"))
    dq_ref, dk_ref, dv_ref, _ = ref.backward(q, k, v, do, w.sm_scale, w.causal)
    tol = GRAD_TOL[w.dtype]
    for name, r in (("dq", dq_ref), ("dk", dk_ref), ("dv", dv_ref)):
        g = head(grads[name], w, b, h)
        assert np.isfinite(g).all(), f"non-finite {name} at head {(b, h)}"
        err = np.abs(g - r)
        scale = max(1.0, float(np.abs(r).max()))
        excess = (err - half_ulp(r, w.dtype)) / scale
        stats["max_" + name] = max(stats.get("max_" + name, 0.0), float(err.max()))
        stats["max_rel_" + name] = max(stats.get("max_rel_" + name, -1.0), float(excess.max()))
        if excess.max() > tol:
            i = np.unravel_index(np.argmax(excess), excess.shape)
            raise AssertionError(f"{name} mismatch at head {(b, h)} row {i[0]} col {i[1]}: gpu {g[i]} ref {r[i]} "
                                 f"(scale {scale:.3g}, tol {tol})")
