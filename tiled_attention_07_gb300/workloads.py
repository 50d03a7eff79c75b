"""Seeded synthetic attention workloads shared by the CUDA path and the oracle.

This module holds no attention arithmetic: only the workload shapes and a
seeded generator of Q, K, V (and dO) tensors.  Both sides of every parity test
draw their inputs from here, so the oracle and the CUDA library see exactly the
same low-precision bits.

Shapes and distributions follow the pages' own workloads:

* "Understanding Triton Tutorials Part 2", section "Fused Attention 2": inputs
  ``[Z, H, N_CTX, HEAD_DIM]`` drawn from N(0, 0.5^2), ``sm_scale = 0.5``,
  ``dout = randn_like(q)``.
* "BUG in flash attention kernel" (triton issue 2626), ``test_op``: the
  ``[seq, heads, d]`` layout with ``q_ctx != seqlen`` (cross attention), seed
  20, N(0, 0.5^2), ``sm_scale = 0.5``.
* "[CS336] Assignment 2: Systems", end-to-end benchmark table: model widths
  768/12 heads, 1280/20 heads and 2560/32 heads, i.e. head dims 64 and 80,
  batch 4, causal attention with ``1/sqrt(d)`` scaling.

Layouts
-------
``"bhsd"``: ``[B, H, seq, d]`` contiguous.
``"shd"``:  ``[seq, heads, d]`` contiguous (batch 1).
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str          # "fp16" | "bf16"
    layout: str         # "bhsd" | "shd"
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    sm_scale: float
    std: float          # standard deviation of q, k, v
    seed: int
    backward: bool = False   # the workload also runs the backward pass

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    def shape(self, n: int):
        if self.layout == "bhsd":
            return (self.B, self.H, n, self.d)
        if self.layout == "shd":
            assert self.B == 1
            return (n, self.H, self.d)
        raise ValueError(self.layout)

    # ---- work accounting (definitions, not arithmetic of the method) ----
    def pairs(self) -> float:
        """Number of (query, key) score entries the method must evaluate."""
        full = float(self.B) * self.H * self.Nq * self.Nk
        return full * 0.5 if self.causal else full

    def fwd_flops(self) -> float:
        """4*B*H*Nq*Nk*d, halved for causal (two GEMMs: QK^T and PV)."""
        return 4.0 * self.pairs() * self.d

    def bwd_flops(self) -> float:
        """10*B*H*Nq*Nk*d, halved for causal (five GEMMs of the recompute backward)."""
        return 10.0 * self.pairs() * self.d

    def fwd_bytes(self) -> float:
        e = 2
        return e * self.d * self.B * self.H * (2 * self.Nq + 2 * self.Nk) + 4.0 * self.B * self.H * self.Nq

    def bwd_bytes(self) -> float:
        e = 2
        return e * self.d * self.B * self.H * (4 * self.Nq + 4 * self.Nk) + 8.0 * self.B * self.H * self.Nq


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("fp16_h1_n128_d64", "fp16", "shd", 1, 1, 128, 128, 64, False, 0.5, 0.5, 20),
        Workload("fp16_h16_nq1000_nk2500_d80", "fp16", "shd", 1, 16, 1000, 2500, 80, False, 0.5, 0.5, 21),
        Workload("bf16_b4_h12_n512_d64_causal", "bf16", "bhsd", 4, 12, 512, 512, 64, True, 1.0 / math.sqrt(64), 1.0, 22),
        Workload("bf16_b4_h20_n4096_d64_causal", "bf16", "bhsd", 4, 20, 4096, 4096, 64, True, 1.0 / math.sqrt(64), 1.0, 23),
        Workload("bf16_b4_h32_n8192_d80_causal_fwdbwd", "bf16", "bhsd", 4, 32, 8192, 8192, 80, True, 1.0 / math.sqrt(80), 1.0, 24,
                 backward=True),
    ]
}

#: The workload one bench step runs: the only one that takes the whole path
#: (forward and backward).
BENCH_WORKLOAD = "bf16_b4_h32_n8192_d80_causal_fwdbwd"


def custom(dtype: str, layout: str, B: int, H: int, Nq: int, Nk: int, d: int, causal: bool,
           sm_scale: Optional[float] = None, std: float = 1.0, seed: int = 0, backward: bool = False) -> Workload:
    """A workload outside the named table (edge cases, sweeps)."""
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    name = f"{dtype}_{layout}_b{B}_h{H}_nq{Nq}_nk{Nk}_d{d}{'_causal' if causal else ''}"
    return Workload(name, dtype, layout, B, H, Nq, Nk, d, causal, float(sm_scale), std, seed, backward)


def make_inputs(w: Workload, device: str = "cpu", with_grad_output: Optional[bool] = None) -> Dict[str, torch.Tensor]:
    """Seeded q, k, v (and dO) in the workload's dtype and layout.

    Values are drawn in fp32 from N(0, std^2) (dO from N(0, 1)) with a CPU
    ``torch.Generator`` seeded by ``w.seed`` and rounded to the dtype (round to
    nearest even), then moved to ``device``.  The same seed always gives the
    same bits.
    """
    if with_grad_output is None:
        with_grad_output = w.backward
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    dt = w.torch_dtype
    out = {}
    for name, n in (("q", w.Nq), ("k", w.Nk), ("v", w.Nk)):
        t = torch.randn(w.shape(n), generator=g, dtype=torch.float32)
        if w.std != 1.0:
            t.mul_(w.std)
        out[name] = t.to(dt)
    if with_grad_output:
        out["do"] = torch.randn(w.shape(w.Nq), generator=g, dtype=torch.float32).to(dt)
    if device != "cpu":
        out = {k: t.to(device) for k, t in out.items()}
    return out


def fp8v_inputs(w: Workload, device: str = "cpu", ld: Optional[int] = None, pad_code: int = 0) -> Dict[str, torch.Tensor]:
    """q, k of ``make_inputs`` and its V stored for the e5m2 path: transposed
    to ``[B, H, d, Nk]``, cast to float8 e5m2 by torch (round to nearest even)
    and held as raw codes (uint8) in rows of ``ld`` bytes (default Nk rounded
    up to 16), the bytes past Nk set to ``pad_code``.  Returns q, k, ``vt``
    (uint8 [B, H, d, ld]) and ``v8`` (the same V values, float32 [B, H, Nk, d])."""
    if w.layout != "bhsd":
        raise ValueError("the e5m2 V path takes the [B, H, seq, d] layout")
    x = make_inputs(w, "cpu", with_grad_output=False)
    if ld is None:
        ld = (w.Nk + 15) // 16 * 16
    codes = x["v"].float().transpose(-1, -2).contiguous().to(torch.float8_e5m2).view(torch.uint8)
    vt = torch.full((w.B, w.H, w.d, ld), pad_code, dtype=torch.uint8)
    vt[..., : w.Nk] = codes
    out = {"q": x["q"], "k": x["k"], "vt": vt,
           "v8": codes.view(torch.float8_e5m2).float().transpose(-1, -2).contiguous()}
    if device != "cpu":
        out = {k: t.to(device) for k, t in out.items()}
    return out


def head_view(t: torch.Tensor, layout: str, b: int, h: int) -> torch.Tensor:
    """The ``[seq, d]`` matrix of one (batch, head) pair."""
    if layout == "bhsd":
        return t[b, h]
    if layout == "shd":
        assert b == 0
        return t[:, h, :]
    raise ValueError(layout)


def stat_view(t: torch.Tensor, layout: str, b: int, h: int) -> torch.Tensor:
    """The ``[Nq]`` row of a per-row statistic (LSE) stored as ``[B, H, Nq]``."""
    return t[b, h]


# ---------------------------------------------------------------------------
# row softmax ("Puzzles 8 Long Softmax") inputs
# ---------------------------------------------------------------------------

SOFTMAX_DTYPES = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class SoftmaxWorkload:
    name: str
    dtype: str      # "fp32" | "fp16" | "bf16"
    rows: int
    T: int
    std: float      # logits ~ N(0, std^2)
    seed: int

    def bytes_moved(self) -> float:
        """Algorithmic HBM bytes: every element read once and written once."""
        e = torch.empty((), dtype=SOFTMAX_DTYPES[self.dtype]).element_size()
        return 2.0 * e * self.rows * self.T


SOFTMAX_WORKLOADS: Dict[str, SoftmaxWorkload] = {
    w.name: w
    for w in [
        # the puzzle's own scale: a handful of rows, T not a tile multiple
        SoftmaxWorkload("fp32_rows4_t200", "fp32", 4, 200, 1.0, 30),
        # long rows: 4096 x 32768 float32 (512 MB each way), two slices per row
        SoftmaxWorkload("fp32_rows4096_t32768", "fp32", 4096, 32768, 3.0, 31),
        # very long rows: 16 rows of 1M bf16 logits (streamed, eight CTAs per row)
        SoftmaxWorkload("bf16_rows16_t1048576", "bf16", 16, 1 << 20, 3.0, 32),
    ]
}


def softmax_inputs(rows: int, T: int, dtype: str, std: float, seed: int, row_stride: Optional[int] = None,
                   device: str = "cpu") -> torch.Tensor:
    """Seeded [rows, T] logits drawn in fp32 from N(0, std^2) with a CPU
    generator and rounded to the dtype; with ``row_stride`` the rows sit in
    a wider buffer (the returned tensor is a view of its first T columns)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn((rows, T), generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    x = x.to(SOFTMAX_DTYPES[dtype])
    if row_stride is not None and row_stride != T:
        buf = torch.zeros((rows, row_stride), dtype=x.dtype)
        buf[:, :T] = x
        if device != "cpu":
            buf = buf.to(device)   # moved whole: a view would be copied densely
        return buf[:, :T]
    return x.to(device) if device != "cpu" else x
