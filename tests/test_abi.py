"""The C ABI library loads, exports every symbol include/fa.h declares, and
rejects bad arguments before touching the GPU (these calls make no CUDA call,
so they run on a machine without a GPU)."""

import ctypes
import os
import re

import pytest
import torch

from tiled_attention_07_gb300 import fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


def header_symbols():
    text = open(HEADER).read()
    return re.findall(r"FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", text)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fa.LIB_PATH):
        from tiled_attention_07_gb300 import build
        build.build()
    return fa.lib()


@pytest.fixture(scope="module")
def L(lib):
    # The argument checks below pass fake device addresses.  Should a check
    # ever let one through, a launch would follow, so these run only where no
    # GPU is visible.
    if torch.cuda.is_available():
        pytest.skip("fake device addresses: argument checks run on a machine without a GPU")
    return lib


def test_header_declares_the_binding_symbols():
    syms = header_symbols()
    assert sorted(syms) == sorted(fa.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for s in header_symbols():
        assert hasattr(lib, s), f"libfa.so does not export {s}"


def test_status_strings_and_version(lib):
    assert fa.fa_version() == "0.1.0"
    for code in range(6):
        assert fa.fa_status_string(code).startswith("FA_")
    assert "unknown" in fa.fa_status_string(99)


def test_workspace_bytes(lib):
    assert fa.fa_bwd_workspace_bytes(4, 32, 8192, 8192, 80) == 2 * 4 * 4 * 32 * 8192
    assert fa.fa_bwd_workspace_bytes(1, 16, 1000, 2500, 80) == 2 * 4 * 16 * 1024
    assert fa.fa_bwd_workspace_bytes(0, 16, 1000, 2500, 80) == 0
    assert fa.fa_bwd_workspace_bytes(2, 3, 0, 5, 64) == 0


FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced here


def fwd(L, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, Nq=128, Nk=128, d=64, scale=0.125, causal=0,
        dtype=fa.FA_BF16):
    return L.fa_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=32), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=7), fa.FA_ERR_UNSUPPORTED),
    (dict(Nk=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nq=-1), fa.FA_ERR_INVALID_ARG),
    (dict(B=-2), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(causal=2), fa.FA_ERR_INVALID_ARG),
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(o=None), fa.FA_ERR_INVALID_ARG),
    (dict(lse=None), fa.FA_ERR_INVALID_ARG),
    (dict(k=FAKE + 8), fa.FA_ERR_INVALID_ARG),
    (dict(lse=FAKE + 4), fa.FA_ERR_INVALID_ARG),
])
def test_fwd_rejects_bad_arguments(L, kw, code):
    assert fwd(L, **kw) == code


def fwd8(L, q=FAKE, k=FAKE, vt=FAKE, o=FAKE, lse=FAKE, B=1, H=1, Nq=128, Nk=128, d=64, ld=128, scale=0.125,
         causal=0, dtype=fa.FA_FP16):
    return L.fa_fwd_fp8v(q, k, vt, o, lse, B, H, Nq, Nk, d, ld, scale, causal, dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=fa.FA_FP32), fa.FA_ERR_UNSUPPORTED),
    (dict(Nk=100, ld=100), fa.FA_ERR_INVALID_ARG),   # row stride not a multiple of 16 bytes
    (dict(Nk=128, ld=112), fa.FA_ERR_INVALID_ARG),   # rows shorter than Nk
    (dict(vt=None), fa.FA_ERR_INVALID_ARG),
    (dict(vt=FAKE + 8), fa.FA_ERR_INVALID_ARG),
    (dict(q=FAKE + 2), fa.FA_ERR_INVALID_ARG),
    (dict(lse=None), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(Nk=0, ld=16), fa.FA_ERR_INVALID_ARG),
])
def test_fwd_fp8v_rejects_bad_arguments(L, kw, code):
    assert fwd8(L, **kw) == code


def test_fwd_fp8v_empty_problems_are_noops(L):
    assert fwd8(L, B=0) == fa.FA_OK
    assert fwd8(L, Nq=0, q=None, o=None, lse=None) == fa.FA_OK


def test_fwd_empty_problems_are_noops(L):
    assert fwd(L, B=0) == fa.FA_OK
    assert fwd(L, H=0) == fa.FA_OK
    assert fwd(L, Nq=0) == fa.FA_OK
    assert fwd(L, Nq=0, q=None, o=None, lse=None) == fa.FA_OK


def test_strided_rejects_bad_strides(L):
    lay = fa.Layout()
    for n in ("q", "k", "v", "o"):
        setattr(lay, n, fa.Strides(128 * 64, 128 * 64, 64))
    args = [FAKE] * 5 + [1, 1, 128, 128, 64, 0.125, 0, fa.FA_BF16]
    lay.k = fa.Strides(128 * 64, 128 * 64, 60)   # 120-byte rows: not a multiple of 16
    assert L.fa_fwd_strided(*args, ctypes.byref(lay), None) == fa.FA_ERR_INVALID_ARG
    lay.k = fa.Strides(128 * 64, 0, 64)
    assert L.fa_fwd_strided(*args, ctypes.byref(lay), None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_strided(*args, None, None) == fa.FA_ERR_INVALID_ARG


def bwd(L, ws=FAKE, ws_bytes=1 << 30, d=64, Nk=128, **kw):
    ptrs = [FAKE] * 9
    return L.fa_bwd(*ptrs, 1, 1, 128, Nk, d, 0.125, 0, fa.FA_BF16, ws, ws_bytes, None)


def test_bwd_phase_rejects_unknown_phase(L):
    ptrs = [FAKE] * 9
    for phase in (0, 4, -1):
        assert L.fa_bwd_phase(phase, *ptrs, 1, 1, 128, 128, 64, 0.125, 0, fa.FA_BF16, None, FAKE, 1 << 20,
                              None) == fa.FA_ERR_INVALID_ARG


def test_bwd_checks_workspace_and_args(L):
    # below the two-pass size is too small for every path (a workspace of the
    # fused size less a little only makes AUTO take the two-pass path)
    need = fa.fa_bwd_workspace_bytes_path(1, 1, 128, 128, 64, fa.FA_BWD_PATH_TWO_PASS)
    assert bwd(L, ws=None) == fa.FA_ERR_WORKSPACE
    assert bwd(L, ws_bytes=need - 16) == fa.FA_ERR_WORKSPACE
    assert bwd(L, d=80, ws_bytes=fa.fa_bwd_workspace_bytes(1, 1, 128, 128, 80) - 16) == fa.FA_ERR_WORKSPACE
    assert bwd(L, ws=FAKE + 4) == fa.FA_ERR_WORKSPACE
    assert bwd(L, d=100) == fa.FA_ERR_UNSUPPORTED
    assert bwd(L, Nk=0) == fa.FA_ERR_INVALID_ARG


def test_inject_rejects_zero_code(L):
    assert L.fa_inject_device_error(0) == fa.FA_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.attention_forward(q, q, q, 0.125, False)


def test_split_workspace_bytes(lib):
    # float32 O_s (d columns) and lse_s per split, rows padded to 128-row tiles
    assert fa.fa_fwd_split_workspace_bytes(1, 16, 1000, 80, 4) == 4 * 4 * 16 * 1024 * 81
    assert fa.fa_fwd_split_workspace_bytes(4, 12, 512, 64, 2) == 4 * 2 * 48 * 512 * 65
    assert fa.fa_fwd_split_workspace_bytes(1, 16, 1000, 80, 1) == 0
    assert fa.fa_fwd_split_workspace_bytes(0, 16, 1000, 80, 4) == 0
    assert fa.fa_fwd_split_workspace_bytes(1, 16, 0, 80, 4) == 0


def test_split_count_without_a_device_is_one(L):
    if torch.cuda.is_available():
        pytest.skip("the count depends on the device's SMs")
    assert fa.fa_fwd_split_count(1, 16, 1000, 2500, 80, False) == 1


def split(L, n_splits=4, ws=FAKE, ws_bytes=1 << 30, layout=None, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, Nq=128, Nk=1024, d=64, scale=0.125, causal=0,
             dtype=fa.FA_BF16)
    a.update(kw)
    return L.fa_fwd_split(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"], a["Nk"], a["d"],
                          a["scale"], a["causal"], a["dtype"], layout, n_splits, ws, ws_bytes, None)


def test_split_checks_count_workspace_and_args(L):
    need = fa.fa_fwd_split_workspace_bytes(1, 1, 128, 64, 4)
    assert split(L, n_splits=0) == fa.FA_ERR_INVALID_ARG
    assert split(L, n_splits=-3) == fa.FA_ERR_INVALID_ARG
    assert split(L, n_splits=65) == fa.FA_ERR_INVALID_ARG
    assert split(L, ws=None) == fa.FA_ERR_WORKSPACE
    assert split(L, ws_bytes=need - 16) == fa.FA_ERR_WORKSPACE
    assert split(L, ws=FAKE + 8) == fa.FA_ERR_WORKSPACE
    assert split(L, d=96) == fa.FA_ERR_UNSUPPORTED
    assert split(L, Nk=0) == fa.FA_ERR_INVALID_ARG
    assert split(L, scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert split(L, k=FAKE + 8) == fa.FA_ERR_INVALID_ARG
    # empty problems are no-ops, with or without a workspace
    assert split(L, B=0, ws=None) == fa.FA_OK
    assert split(L, Nq=0, ws=None) == fa.FA_OK
    lay = fa.Layout()
    for n in ("q", "k", "v", "o"):
        setattr(lay, n, fa.Strides(1024 * 64, 1024 * 64, 64))
    lay.v = fa.Strides(1024 * 64, 1024 * 64, 60)   # 120-byte rows
    assert split(L, layout=ctypes.byref(lay)) == fa.FA_ERR_INVALID_ARG


def test_softmax_rows_rejects_bad_arguments(L):
    def sm(x=FAKE, z=FAKE + (1 << 24), lse=None, rows=4, T=100, xs=100, zs=100, dtype=fa.FA_FP32):
        return L.fa_softmax_rows(x, z, lse, rows, T, xs, zs, dtype, None)
    assert sm(dtype=3) == fa.FA_ERR_UNSUPPORTED
    assert sm(T=0) == fa.FA_ERR_INVALID_ARG
    assert sm(rows=-1) == fa.FA_ERR_INVALID_ARG
    assert sm(xs=99) == fa.FA_ERR_INVALID_ARG            # stride shorter than a row
    assert sm(xs=101, zs=101) == fa.FA_ERR_INVALID_ARG   # 404-byte rows: not 16-byte aligned
    assert sm(dtype=fa.FA_BF16, xs=100, zs=100) == fa.FA_ERR_INVALID_ARG   # 200-byte rows
    assert sm(x=None) == fa.FA_ERR_INVALID_ARG
    assert sm(z=FAKE + 8) == fa.FA_ERR_INVALID_ARG
    assert sm(lse=FAKE + 2) == fa.FA_ERR_INVALID_ARG
    assert sm(z=FAKE + 16, T=96) == fa.FA_ERR_INVALID_ARG   # overlapping, not identical
    assert sm(z=FAKE, xs=100, zs=104) == fa.FA_ERR_INVALID_ARG   # same base, other stride
    assert sm(rows=0) == fa.FA_OK


# Sizes whose strides or workspace sizes overflow 64-bit arithmetic are
# rejected, never wrapped into something that passes a check.
I32_MAX = 2 ** 31 - 1
SIZE_MAX = 2 ** 64 - 1


def test_sequence_length_limit(L):
    limit = 1 << 30
    assert fwd(L, Nq=limit + 1) == fa.FA_ERR_INVALID_ARG
    assert fwd(L, Nk=limit + 1) == fa.FA_ERR_INVALID_ARG
    assert fwd(L, Nq=I32_MAX, Nk=I32_MAX) == fa.FA_ERR_INVALID_ARG
    assert fwd8(L, Nq=limit + 1) == fa.FA_ERR_INVALID_ARG
    assert split(L, Nk=limit + 1) == fa.FA_ERR_INVALID_ARG
    ptrs = [FAKE] * 9
    assert L.fa_bwd(*ptrs, 1, 1, limit + 1, 128, 64, 0.125, 0, fa.FA_BF16, FAKE, SIZE_MAX, None) == \
        fa.FA_ERR_INVALID_ARG


def test_contiguous_strides_that_overflow_are_rejected(L):
    # H * Nq * d = 2^30 * 2^30 * 64 elements: no int64 wrap, a stride past 2^40 bytes
    assert fwd(L, B=1, H=1 << 30, Nq=1 << 30, Nk=128) == fa.FA_ERR_INVALID_ARG
    # the batch stride H * Nq * d reaches 2^39 elements (2^40 bytes)
    assert fwd(L, B=2, H=(1 << 39) // (1024 * 64), Nq=1024, Nk=128) == fa.FA_ERR_INVALID_ARG


def test_strided_stride_limit(L):
    lay = fa.Layout()
    for n in ("q", "k", "v", "o"):
        setattr(lay, n, fa.Strides(128 * 64, 128 * 64, 64))
    args = [FAKE] * 5 + [2, 1, 128, 128, 64, 0.125, 0, fa.FA_BF16]
    lay.q = fa.Strides(1 << 39, 128 * 64, 64)            # 2^40 bytes: past the TMA limit
    assert L.fa_fwd_strided(*args, ctypes.byref(lay), None) == fa.FA_ERR_INVALID_ARG
    lay.q = fa.Strides(2 ** 63 - 8, 128 * 64, 64)        # doubled, wraps negative
    assert L.fa_fwd_strided(*args, ctypes.byref(lay), None) == fa.FA_ERR_INVALID_ARG
    lay.q = fa.Strides(-(1 << 20), 128 * 64, 64)
    assert L.fa_fwd_strided(*args, ctypes.byref(lay), None) == fa.FA_ERR_INVALID_ARG


def test_fp8v_batch_stride_limit(L):
    # V^T batch stride = ld * d * H bytes must stay below 2^40
    ld = 1 << 24
    assert fwd8(L, B=2, H=(1 << 40) // (ld * 64), Nk=128, ld=ld) == fa.FA_ERR_INVALID_ARG
    assert fwd8(L, B=2, H=I32_MAX // 2, Nk=128, ld=(1 << 32) - 16, d=128) == fa.FA_ERR_INVALID_ARG


def test_workspace_sizes_saturate(lib):
    assert fa.fa_bwd_workspace_bytes(I32_MAX, I32_MAX, I32_MAX, 1, 64) == SIZE_MAX
    assert fa.fa_fwd_split_workspace_bytes(I32_MAX, I32_MAX, 1 << 30, 128, 64) == SIZE_MAX
    # no saturation at ordinary sizes
    assert fa.fa_bwd_workspace_bytes(4, 32, 8192, 8192, 80) == 2 * 4 * 4 * 32 * 8192


def test_softmax_span_overflow_is_rejected(L):
    # (rows - 1) * stride * 4 bytes overflows int64
    assert L.fa_softmax_rows(FAKE, FAKE + (1 << 24), None, 1 << 20, 128, 2 ** 45, 2 ** 45, fa.FA_FP32,
                             None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_softmax_rows(FAKE, FAKE + (1 << 24), None, 2, 128, 2 ** 62, 128, fa.FA_FP32,
                             None) == fa.FA_ERR_INVALID_ARG


def test_bwd_path_workspace_bytes(lib):
    rows = 4 * 20 * 4096
    two = fa.fa_bwd_workspace_bytes_path(4, 20, 4096, 4096, 64, fa.FA_BWD_PATH_TWO_PASS)
    fused = fa.fa_bwd_workspace_bytes_path(4, 20, 4096, 4096, 64, fa.FA_BWD_PATH_FUSED)
    assert two == 8 * rows and fused == 4 * (2 + 64) * rows
    # AUTO prefers the fused path at d = 64 and the two-pass path elsewhere
    assert fa.fa_bwd_workspace_bytes(4, 20, 4096, 4096, 64) == fused
    assert fa.fa_bwd_workspace_bytes_path(4, 20, 4096, 4096, 64, fa.FA_BWD_PATH_AUTO) == fused
    assert fa.fa_bwd_workspace_bytes(4, 32, 8192, 8192, 80) == 8 * 4 * 32 * 8192
    for d in (80, 128):
        assert fa.fa_bwd_workspace_bytes_path(1, 2, 300, 300, d, fa.FA_BWD_PATH_FUSED) == 0
    assert fa.fa_bwd_workspace_bytes_path(1, 2, 0, 300, 64, fa.FA_BWD_PATH_FUSED) == 0
    assert fa.fa_bwd_workspace_bytes_path(1, 2, 300, 300, 64, 7) == 0


def test_bwd_ex_rejects_bad_path_phase_and_size(L):
    ptrs = [FAKE] * 9

    def ex(path, phase=0, d=64, ws_bytes=1 << 30):
        return L.fa_bwd_ex(path, phase, *ptrs, 1, 1, 128, 128, d, 0.125, 0, fa.FA_BF16, None, FAKE, ws_bytes, None)

    assert ex(3) == fa.FA_ERR_INVALID_ARG
    assert ex(-1) == fa.FA_ERR_INVALID_ARG
    for phase in (4, -1):
        assert ex(fa.FA_BWD_PATH_FUSED, phase) == fa.FA_ERR_INVALID_ARG
    assert ex(fa.FA_BWD_PATH_FUSED, d=80) == fa.FA_ERR_UNSUPPORTED
    two = fa.fa_bwd_workspace_bytes_path(1, 1, 128, 128, 64, fa.FA_BWD_PATH_TWO_PASS)
    assert ex(fa.FA_BWD_PATH_FUSED, ws_bytes=two) == fa.FA_ERR_WORKSPACE
    assert ex(fa.FA_BWD_PATH_TWO_PASS, ws_bytes=two - 16) == fa.FA_ERR_WORKSPACE
