"""Row-softmax parity: fa_softmax_rows (through the C ABI) against the
float64 oracle, element by element, for each path of the kernel (one CTA per
row, a cluster of CTAs per row, streamed slices), ragged lengths, padded row
strides, in place, and the special values."""

import numpy as np
import pytest
import torch

import oracle.softmax as ref
from tiled_attention_07_gb300 import fa
from tiled_attention_07_gb300 import workloads as W

pytestmark = pytest.mark.gpu

# z: float32 output within a relative 1e-5 of the exact value (exp2
# approximation, float32 sums); 16-bit outputs within half an ulp more.
Z_REL = 1e-5
LSE_ABS = 2e-5


def half_ulp16(ref_vals, dtype):
    """Half the spacing of the 16-bit format at each value, subnormals
    included (their spacing is fixed: 2^-24 for fp16, 2^-133 for bf16)."""
    mant, emin = (7, -126) if dtype == torch.bfloat16 else (10, -14)
    e = np.floor(np.log2(np.maximum(np.abs(ref_vals), 1e-300)))
    return 0.5 * np.exp2(np.maximum(e, emin) - mant)


def check(x, z, lse):
    x64 = x.float().cpu().double().numpy()
    z_ref, lse_ref = ref.softmax_rows(x64)
    z_gpu = z.float().cpu().double().numpy()
    tol = Z_REL * z_ref + 1e-37
    if x.dtype != torch.float32:
        tol = tol + half_ulp16(z_ref, x.dtype)
    err = np.abs(z_gpu - z_ref)
    bad = err > tol
    assert not bad.any(), f"z mismatch at {np.argwhere(bad)[0]}: gpu {z_gpu[bad][0]} ref {z_ref[bad][0]}"
    if lse is not None:
        l_gpu = lse.cpu().double().numpy()
        assert (np.abs(l_gpu - lse_ref) <= LSE_ABS * np.maximum(1.0, np.abs(lse_ref))).all(), "lse mismatch"
    return float((err / np.maximum(z_ref, 1e-30)).max())


def run(x, in_place=False, want_lse=True):
    if in_place:
        z = x
    else:   # same (possibly padded) row stride as x
        rows, T = x.shape
        stride = x.stride(0) if rows > 1 else T
        z = torch.full((rows, stride), float("nan"), dtype=x.dtype, device=x.device)[:, :T]
    lse = torch.full((x.shape[0],), float("nan"), dtype=torch.float32, device=x.device) if want_lse else None
    x_copy = x.clone() if in_place else x
    fa.fa_softmax_rows(x, z, lse)
    torch.cuda.synchronize()
    return x_copy, z, lse


@pytest.mark.parametrize("dtype,rows,T,stride,std", [
    ("fp32", 4, 200, 208, 1.0),          # the puzzle's scale, padded stride
    ("fp32", 1000, 1001, 1004, 3.0),     # ragged T
    ("fp16", 300, 4096, None, 3.0),
    ("bf16", 64, 16384, None, 3.0),      # exactly one slice
    ("fp32", 8, 100003, 100004, 3.0),    # a cluster of 7 CTAs per row, ragged tail
    ("bf16", 5, 131072, None, 5.0),      # a cluster of 8, exactly full
    ("fp32", 3, 1000003, 1000004, 3.0),  # streamed: slices longer than the on-chip buffer
    ("bf16", 1, 7, None, 1.0),           # a single short row
])
def test_parity(dtype, rows, T, stride, std):
    x = W.softmax_inputs(rows, T, dtype, std, seed=rows + T, row_stride=stride, device="cuda")
    x0, z, lse = run(x)
    print(dtype, rows, T, "max rel err", check(x0, z, lse))


def test_named_workload_small():
    w = W.SOFTMAX_WORKLOADS["fp32_rows4_t200"]
    x = W.softmax_inputs(w.rows, w.T, w.dtype, w.std, w.seed, row_stride=208, device="cuda")
    x0, z, lse = run(x)
    check(x0, z, lse)


@pytest.mark.parametrize("name", ["fp32_rows4096_t32768", "bf16_rows16_t1048576"])
def test_named_workload_sampled_rows(name):
    w = W.SOFTMAX_WORKLOADS[name]
    x = W.softmax_inputs(w.rows, w.T, w.dtype, w.std, w.seed, device="cuda")
    _, z, lse = run(x)
    idx = sorted({0, w.rows // 3, w.rows - 1})
    check(x[idx], z[idx], lse[idx])
    # every row sums to one
    assert torch.allclose(z.float().sum(dim=1), torch.ones(w.rows, device="cuda"), atol=2e-3 if w.dtype != "fp32" else 1e-4)


def test_in_place_and_without_lse():
    x = W.softmax_inputs(50, 70000, "fp32", 3.0, seed=5, row_stride=70004, device="cuda")
    x0, z, _ = run(x.clone(), in_place=True, want_lse=False)
    check(x0, z, None)


def test_special_values():
    x = W.softmax_inputs(4, 40000, "fp32", 2.0, seed=6, device="cuda")
    x[0, :] = 1.25                        # constant row: 1/T
    x[1, 123] = 1.0e4                     # one dominating logit
    x[2, 5000:39000] = float("-inf")      # mostly masked, across slices
    x[3, :] += 3.0e4                      # huge logits: the max subtraction
    x0, z, lse = run(x)
    check(x0, z, lse)
    assert torch.all(z[2, 5000:39000] == 0)
