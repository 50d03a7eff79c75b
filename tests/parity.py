"""Helpers for the CUDA-vs-oracle parity tests.

Tolerances (stated for the forward by the workload definition, derived for
the backward):

* forward O: max |O_gpu - O_ref| <= 2e-3 (fp16) / 1e-2 (bf16), where each
  element may in addition be off by half an ulp of the output type at
  |O_ref| (the rounding of a correct result to fp16/bf16 alone reaches
  0.0156 for bf16 values in [4, 8)); the plain max is reported as well.
* forward LSE: max |LSE_gpu - LSE_ref| <= 1e-3.
* backward dQ, dK, dV, two bounds that must both hold:
  (a) per head: max |d_gpu - d_ref| <= tol * max(1, max |d_ref|) with
      tol = 2e-3 (fp16) / 1e-2 (bf16), plus half an output ulp per element;
  (b) per 128-row tile T (the kernels' tile):
      ||d_gpu[T] - d_ref[T]||_F <= 2 ||d_naive[T] - d_ref[T]||_F + floor,
      where d_naive is a plain, unfused computation of the same gradients at
      the library's storage precision (``naive_grads``);
  (c) per row: ||d_gpu[r] - d_ref[r]|| <= 6 sigma_r + ||half ulp(d_ref[r])||
      + floor, sigma_r the standard deviation of the row's error in a
      first-order model of rounding at the input type (``rounding_sigma``).
  floor is 2^-12 of the head's RMS row norm (per row; sqrt(rows) of it per
  tile); the per-tile floor adds a quarter of the rounding model's deviation
  of the tile, so that a tile whose exact gradient vanishes (the naive
  reference then has no error at all) is not failed on rounding noise.  (a) alone scales with the largest gradient of the head and cannot
  see rows far below it.  (b) is the tight check: a tile's error sums
  thousands of independent roundings, so the ratio of two same-precision
  computations stays close to 1, and a 1 % error on one tile fails it.  A
  single row cannot be held to the naive reference's row: query i of a
  causal head sees i + 1 keys and dS sums to zero along the row, so an early
  row of dQ is small and its error is dominated by one random scalar, the
  rounding error of D_i = rowsum(O o dO) (O is stored at the input type),
  which for the naive reference is an independent draw.  (c) therefore uses
  the model's spread instead; it rejects a zeroed, swapped or sign-flipped
  row.
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


#: Factor of the per-tile and per-row bounds against the same-precision
#: naive reference.
NAIVE_FACTOR = 2.0
#: Rows per tile of the per-tile bound (the kernels' 128-row tiles).
TILE_ROWS = 128
#: Unit roundoff of each input type (largest relative error of rounding to
#: nearest), and the per-row bound in standard deviations of the rounding
#: model (a sum of k uniform errors never exceeds sqrt(3 k) of them; many
#: terms are near Gaussian, where 6 deviations are not reached in 10^8 rows).
UNIT_ROUNDOFF = {"fp16": 2.0 ** -11, "bf16": 2.0 ** -8}
ROW_SIGMAS = 6.0
#: Share of the rounding model's deviation added to the per-tile floor.
TILE_SIGMAS = 0.25
#: Absolute floor, relative to the head's RMS row norm (rows whose exact
#: gradient is zero, e.g. dQ of query 0 under the causal mask, where both
#: sides return rounding noise).
ROW_FLOOR = 2.0 ** -12


def naive_grads(q, k, v, do, sm_scale: float, causal: bool, dtype: str):
    """dQ, dK, dV of one head by the plain, unfused computation (S and P
    materialised) at the library's storage precision, for the per-row bound.

    The steps are those of "[CS336] Assignment 2: Systems", "FlashAttention V2
    / High level" (P = exp(S - L), D = rowsum(O o dO), dS = P o (dP - D),
    dV = P^T dO, dQ = sm_scale dS K, dK = sm_scale dS^T Q), in float32 with
    the roundings to the input type that the library makes: P before the
    products with V and dO ("Fused Attention 2" casts p to V's type before
    the product), the forward output O (D is formed from the stored O), dS
    before its products, and the returned gradients.  S stays float32: the
    pages' PyTorch reference rounds S to the input type too, which alone
    costs about 0.5 % per row in bf16 (2.4 % worst) and would make the bound
    too loose to see a 1 % error.  Inputs are float64 arrays holding 16-bit
    values (exact in float32).  dtype "fp32" leaves every rounding out (the
    steps alone, for the checker's own test).
    """
    tdt = torch.float32 if dtype == "fp32" else W.DTYPES[dtype]
    qf, kf, vf, dof = (torch.from_numpy(np.ascontiguousarray(a)).float() for a in (q, k, v, do))
    s = (qf @ kf.T) * sm_scale
    if causal:
        nq, nk = s.shape
        s = s.masked_fill(torch.arange(nk)[None, :] > torch.arange(nq)[:, None], float("-inf"))
    p = torch.exp(s - torch.logsumexp(s, dim=-1, keepdim=True))
    pr = p.to(tdt).float()
    o = (pr @ vf).to(tdt).float()
    dsum = (o * dof).sum(dim=-1, keepdim=True)
    dv = (pr.T @ dof).to(tdt)
    ds = (p * (dof @ vf.T - dsum)).to(tdt).float()
    dq = (sm_scale * (ds @ kf)).to(tdt)
    dk = (sm_scale * (ds.T @ qf)).to(tdt)
    return tuple(t.double().numpy() for t in (dq, dk, dv))


def rounding_sigma(q, k, v, do, sm_scale: float, causal: bool, dtype: str):
    """Per-row standard deviation of dQ's, dK's and dV's error in a
    first-order model of computing them at the input type's precision.

    Each rounding to the input type is taken as an independent error uniform
    in [-u |x|, u |x|] (variance u^2 x^2 / 3, u the unit roundoff); float32
    arithmetic is exact at this order.  The roundings, and what they reach:
    * P before the products with V (forward) and dO (dV): dV_j gets
      sum_i dP_ij dO_i;
    * O, stored at the input type, and the forward's P: D_i = rowsum(O o dO)
      gets dD_i = sum_d (dO_O + sum_j dP_ij V_jd) dO_id, and dS_ij = P_ij
      (dP_ij - D_i) gets -P_ij dD_i;
    * dS before its products: dQ_i gets sm_scale sum_j d(dS_ij) K_j, dK_j
      gets sm_scale sum_i d(dS_ij) Q_i, besides the dD terms.
    The output rounding is left out (the bound adds half an ulp of the
    result).  The steps are those of "[CS336] Assignment 2: Systems",
    "FlashAttention V2 / High level"; the intermediates are taken in float32.
    Returns three float64 arrays (dq rows, dk rows, dv rows).
    """
    var_u = UNIT_ROUNDOFF[dtype] ** 2 / 3.0
    qf, kf, vf, dof = (torch.from_numpy(np.ascontiguousarray(a)).float() for a in (q, k, v, do))
    s = (qf @ kf.T) * sm_scale
    if causal:
        nq, nk = s.shape
        s = s.masked_fill(torch.arange(nk)[None, :] > torch.arange(nq)[:, None], float("-inf"))
    p = torch.exp(s - torch.logsumexp(s, dim=-1, keepdim=True))
    o = p @ vf
    ds = p * (dof @ vf.T - (o * dof).sum(dim=-1, keepdim=True))
    p2 = p * p
    var_d = var_u * (dof * dof * (o * o + p2 @ (vf * vf))).sum(dim=-1)          # [Nq]
    var_dv = var_u * (p2.T @ (dof * dof))
    ds2 = ds * ds
    sc2 = float(sm_scale) ** 2
    var_dq = sc2 * (var_u * (ds2 @ (kf * kf)) + var_d[:, None] * (p @ kf) ** 2)
    var_dk = sc2 * (var_u * (ds2.T @ (qf * qf)) + (p2 * var_d[:, None]).T @ (qf * qf))
    return tuple(torch.sqrt(t.sum(dim=-1)).double().numpy() for t in (var_dq, var_dk, var_dv))


def check_grads(dtype: str, got: dict, ref: dict, naive: dict, where, stats: dict, sigma: dict):
    """The three backward bounds (module docstring) for one head: got, ref,
    naive map "dq", "dk", "dv" to float64 [rows, d] arrays, sigma to the
    per-row deviations of ``rounding_sigma``.  Raises AssertionError naming
    the first failing tensor, rows or row."""
    tol = GRAD_TOL[dtype]
    for name in ("dq", "dk", "dv"):
        g, r, n = got[name], ref[name], naive[name]
        assert np.isfinite(g).all(), f"non-finite {name} at {where}"
        err = np.abs(g - r)
        scale = max(1.0, float(np.abs(r).max()))
        excess = (err - half_ulp(r, dtype)) / scale
        stats["max_" + name] = max(stats.get("max_" + name, 0.0), float(err.max()))
        stats["max_rel_" + name] = max(stats.get("max_rel_" + name, -1.0), float(excess.max()))
        if excess.max() > tol:
            i = np.unravel_index(np.argmax(excess), excess.shape)
            raise AssertionError(f"{name} mismatch at {where} row {i[0]} col {i[1]}: gpu {g[i]} ref {r[i]} "
                                 f"(scale {scale:.3g}, tol {tol})")
        e2_row = np.sum((g - r) ** 2, axis=1)
        n2_row = np.sum((n - r) ** 2, axis=1)
        floor = ROW_FLOOR * float(np.sqrt(np.mean(np.sum(r * r, axis=1))))
        # (b) per tile
        rows = g.shape[0]
        for t0 in range(0, rows, TILE_ROWS):
            sl = slice(t0, min(rows, t0 + TILE_ROWS))
            e_t = float(np.sqrt(e2_row[sl].sum()))
            n_t = float(np.sqrt(n2_row[sl].sum()))
            f_t = floor * np.sqrt(sl.stop - sl.start) + TILE_SIGMAS * float(np.sqrt(np.sum(sigma[name][sl] ** 2)))
            stats["max_tile_frac_" + name] = max(stats.get("max_tile_frac_" + name, 0.0),
                                                 e_t / max(NAIVE_FACTOR * n_t + f_t, 1e-300))
            if e_t > NAIVE_FACTOR * n_t + f_t:
                raise AssertionError(f"{name} rows [{sl.start}, {sl.stop}) at {where}: |gpu - ref| = {e_t:.3g} > "
                                     f"{NAIVE_FACTOR} x naive error {n_t:.3g} + floor {f_t:.3g}")
        # (c) per row
        e_row = np.sqrt(e2_row)
        ulp_row = np.linalg.norm(half_ulp(r, dtype), axis=1)
        bound = ROW_SIGMAS * sigma[name] + ulp_row + floor
        stats["max_row_frac_" + name] = max(stats.get("max_row_frac_" + name, 0.0),
                                            float((e_row / np.maximum(bound, 1e-300)).max()))
        bad = e_row > bound
        if bad.any():
            i = int(np.argmax(e_row - bound))
            raise AssertionError(f"{name} row {i} at {where}: |gpu - ref| = {e_row[i]:.3g} > {ROW_SIGMAS} x "
                                 f"rounding sigma {sigma[name][i]:.3g} + half ulps {ulp_row[i]:.3g} + floor "
                                 f"{floor:.3g} (|ref row| = {float(np.linalg.norm(r[i])):.3g}; "
                                 f"{int(bad.sum())} rows fail)")


def check_bwd_head(w: W.Workload, x: dict, grads: dict, b: int, h: int, stats: dict):
    q, k, v, do = (head(x[n], w, b, h) for n in ("q", "k", "v", "do"))
    dq_ref, dk_ref, dv_ref, _ = ref.backward(q, k, v, do, w.sm_scale, w.causal)
    nv = naive_grads(q, k, v, do, w.sm_scale, w.causal, w.dtype)
    sg = rounding_sigma(q, k, v, do, w.sm_scale, w.causal, w.dtype)
    got = {name: head(grads[name], w, b, h) for name in ("dq", "dk", "dv")}
    check_grads(w.dtype, got, {"dq": dq_ref, "dk": dk_ref, "dv": dv_ref}, dict(zip(("dq", "dk", "dv"), nv)),
                (b, h), stats, dict(zip(("dq", "dk", "dv"), sg)))
