"""What the Python binding hands the C ABI: pointers, sizes, strides and
workspace, checked on CPU against a stand-in library that records each call.
The CUDA-only gates (device check, device context, current stream) are
replaced for the test, so CPU tensors pass through the same marshalling a
GPU call takes."""

import contextlib
import ctypes

import pytest
import torch

from tiled_attention_07_gb300 import fa

BF = torch.bfloat16


class FakeLib:
    def __init__(self, ws_bytes=4096):
        self.calls = []
        self.ws_bytes = ws_bytes

    def __getattr__(self, name):
        def call(*args):
            self.calls.append((name, args))
            return self.ws_bytes if name.endswith("workspace_bytes") else fa.FA_OK
        return call


@pytest.fixture
def lib(monkeypatch):
    L = FakeLib()
    monkeypatch.setattr(fa, "_lib", L)
    monkeypatch.setattr(fa, "_check_cuda", lambda *ts: None)
    monkeypatch.setattr(fa, "_stream", lambda stream, device=None: 7)
    monkeypatch.setattr(fa.torch.cuda, "device", lambda d: contextlib.nullcontext())
    return L


def last(L, name):
    calls = [a for n, a in L.calls if n == name]
    assert calls, f"{name} not called; calls: {[n for n, _ in L.calls]}"
    return calls[-1]


def strides(s):
    return (s.b, s.h, s.s)


def test_contiguous_forward(lib):
    q, k, v = torch.zeros(2, 3, 130, 64, dtype=BF), torch.zeros(2, 3, 300, 64, dtype=BF), torch.zeros(2, 3, 300, 64, dtype=BF)
    o, lse = torch.zeros_like(q), torch.zeros(2, 3, 130)
    fa.fa_fwd(q, k, v, o, lse, 0.125, True)
    a = last(lib, "fa_fwd")
    assert a[:5] == (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr())
    assert a[5:10] == (2, 3, 130, 300, 64)
    assert a[10] == pytest.approx(0.125) and a[11] == 1 and a[12] == fa.FA_BF16 and a[13] == 7


def test_seq_heads_d_forward_uses_strides(lib):
    Nq, Nk, H, d = 100, 250, 4, 80
    q, k, v = torch.zeros(Nq, H, d, dtype=torch.float16), torch.zeros(Nk, H, d, dtype=torch.float16), \
        torch.zeros(Nk, H, d, dtype=torch.float16)
    o, lse = torch.zeros_like(q), torch.zeros(1, H, Nq)
    fa.fa_fwd(q, k, v, o, lse, 0.5, False)
    a = last(lib, "fa_fwd_strided")
    assert a[5:10] == (1, H, Nq, Nk, d) and a[12] == fa.FA_FP16
    lay = a[13]._obj
    assert strides(lay.q) == (Nq * H * d, d, H * d)
    assert strides(lay.k) == (Nk * H * d, d, H * d)
    assert strides(lay.o) == (Nq * H * d, d, H * d)


def test_permuted_view_forward_uses_strides(lib):
    B, S, H, d = 2, 256, 4, 64
    base = [torch.zeros(B, S, H, d, dtype=BF) for _ in range(4)]
    q, k, v, o = (t.transpose(1, 2) for t in base)      # [B, H, S, d] views of [B, S, H, d]
    fa.fa_fwd(q, k, v, o, torch.zeros(B, H, S), 0.125, False)
    lay = last(lib, "fa_fwd_strided")[13]._obj
    for n in ("q", "k", "v", "o"):
        assert strides(getattr(lay, n)) == (S * H * d, d, H * d)


def test_backward_pointer_order_and_workspace(lib):
    B, H, Nq, Nk, d = 1, 2, 128, 200, 64
    q, o, do, dq = (torch.zeros(B, H, Nq, d, dtype=BF) for _ in range(4))
    k, v, dk, dv = (torch.zeros(B, H, Nk, d, dtype=BF) for _ in range(4))
    lse = torch.zeros(B, H, Nq)
    ws = torch.zeros(5000, dtype=torch.uint8)
    fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, 0.125, True, ws)
    a = last(lib, "fa_bwd")
    assert a[:9] == tuple(t.data_ptr() for t in (q, k, v, o, do, lse, dq, dk, dv))
    assert a[9:14] == (B, H, Nq, Nk, d) and a[15] == 1 and a[16] == fa.FA_BF16
    assert a[17] == ws.data_ptr() and a[18] == 5000 and a[19] == 7


def test_backward_allocates_the_workspace_it_asks_for(lib):
    q, o, do, dq = (torch.zeros(1, 1, 128, 64, dtype=BF) for _ in range(4))
    k, v, dk, dv = (torch.zeros(1, 1, 128, 64, dtype=BF) for _ in range(4))
    fa.fa_bwd(q, k, v, o, do, torch.zeros(1, 1, 128), dq, dk, dv, 0.125, False)
    assert last(lib, "fa_bwd_workspace_bytes") == (1, 1, 128, 128, 64)
    assert last(lib, "fa_bwd")[18] == lib.ws_bytes


def test_backward_phase(lib):
    q, o, do, dq = (torch.zeros(1, 2, 64, 80, dtype=BF) for _ in range(4))
    k, v, dk, dv = (torch.zeros(1, 2, 96, 80, dtype=BF) for _ in range(4))
    ws = torch.zeros(1024, dtype=torch.uint8)
    fa.fa_bwd_phase(fa.FA_BWD_DQ, q, k, v, o, do, torch.zeros(1, 2, 64), dq, dk, dv, 0.1, True, ws)
    a = last(lib, "fa_bwd_phase")
    assert a[0] == fa.FA_BWD_DQ and a[10:15] == (1, 2, 64, 96, 80) and a[18] is None and a[19] == ws.data_ptr() and a[20] == 1024


def test_split_forward(lib):
    q, o = torch.zeros(1, 16, 1000, 80, dtype=torch.float16), torch.zeros(1, 16, 1000, 80, dtype=torch.float16)
    k, v = torch.zeros(1, 16, 2500, 80, dtype=torch.float16), torch.zeros(1, 16, 2500, 80, dtype=torch.float16)
    ws = torch.zeros(256, dtype=torch.float32)
    fa.fa_fwd_split(q, k, v, o, torch.zeros(1, 16, 1000), 0.5, False, 4, ws)
    a = last(lib, "fa_fwd_split")
    assert a[5:10] == (1, 16, 1000, 2500, 80) and a[14] == 4 and a[15] == ws.data_ptr() and a[16] == 1024
    assert strides(a[13]._obj.k) == (16 * 2500 * 80, 2500 * 80, 80)


def test_fp8v_forward_passes_the_row_length(lib):
    B, H, Nq, Nk, d, ld = 1, 2, 128, 200, 64, 208
    q, o = torch.zeros(B, H, Nq, d, dtype=BF), torch.zeros(B, H, Nq, d, dtype=BF)
    k = torch.zeros(B, H, Nk, d, dtype=BF)
    vt = torch.zeros(B, H, d, ld, dtype=torch.uint8)[..., :Nk]
    fa.fa_fwd_fp8v(q, k, vt, o, torch.zeros(B, H, Nq), 0.125, True)
    a = last(lib, "fa_fwd_fp8v_ex")
    assert a[2] == vt.data_ptr() and a[5:11] == (B, H, Nq, Nk, d, ld) and a[14] == fa.FA_FP8V_PAGE_STEPS
    fa.fa_fwd_fp8v(q, k, vt, o, torch.zeros(B, H, Nq), 0.125, True, mode=fa.FA_FP8V_LAZY_MAX)
    assert last(lib, "fa_fwd_fp8v_ex")[14] == fa.FA_FP8V_LAZY_MAX


def test_softmax_rows_strides(lib):
    x = torch.zeros(6, 112)[:, :100]
    z = torch.zeros(6, 100)
    fa.fa_softmax_rows(x, z)
    a = last(lib, "fa_softmax_rows")
    assert a[3:7] == (6, 100, 112, 100) and a[2] is None and a[7] == fa.FA_FP32
    # one row: its stride is never used, so the smallest valid one is passed
    fa.fa_softmax_rows(torch.zeros(1, 100, dtype=BF), torch.zeros(1, 100, dtype=BF))
    assert last(lib, "fa_softmax_rows")[5:7] == (104, 104)
